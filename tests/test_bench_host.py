"""Host-side arithmetic of the benchmark (no GPU): the algorithmic bytes behind every GB/s figure.

Decode reads each packed word, scale and zero once plus the activations; the grouped (mixture of
experts) layer reads the whole weight of every expert that holds rows and nothing of the others."""
import numpy as np

import bench
import gptq_inputs


def test_decode_bytes_of_the_llama_workload():
    wl = gptq_inputs.WORKLOADS["llama7b_decode_4bit_g128"]
    # qweight 512 x 11008 words + scales 32 x 11008 halves + qzeros 32 x 1376 words + A 4096 halves
    assert bench.algorithmic_bytes(wl, 1) == 512 * 11008 * 4 + 32 * 11008 * 2 + 32 * 1376 * 4 + 4096 * 2
    assert bench.algorithmic_bytes(wl, 1) == 23_433_216


def test_act_order_bytes_include_g_idx():
    wl = gptq_inputs.WORKLOADS["act_order_3bit_g128"]
    plain = bench.algorithmic_bytes(wl, 16)
    assert plain == 480 * 13824 * 4 + 40 * 13824 * 2 + 40 * 1296 * 4 + 16 * 5120 * 2 + 5120 * 4


def test_grouped_bytes_count_only_routed_experts():
    mw = gptq_inputs.MOE_WORKLOADS["moe_mixtral_4bit_g128"]
    per_expert = 512 * 14336 * 4 + 32 * 14336 * 2 + 32 * 1792 * 4
    for T in mw.Ts:
        r = gptq_inputs.draw_routing(mw, T)
        active = len(set(np.flatnonzero(np.diff(r.offsets))))
        nbytes, counted = bench.grouped_bytes(mw, r.offsets)
        assert counted == active
        assert nbytes == active * per_expert + T * mw.topk * mw.K * 2 + (mw.E + 1) * 4
    # no expert holds rows: only the offsets are read
    assert bench.grouped_bytes(mw, np.zeros(mw.E + 1, np.int32)) == ((mw.E + 1) * 4, 0)


def test_routing_is_a_valid_grouping():
    mw = gptq_inputs.MOE_WORKLOADS["moe_mixtral_4bit_g128"]
    for T in (1, 8, 33):
        r = gptq_inputs.draw_routing(mw, T)
        assert r.offsets[0] == 0 and r.offsets[-1] == T * mw.topk
        assert np.all(np.diff(r.offsets) >= 0)
        # each token appears topk times, never twice for one expert
        assert np.array_equal(np.bincount(r.row_token, minlength=T), np.full(T, mw.topk))
        for e in range(mw.E):
            toks = r.row_token[r.offsets[e]:r.offsets[e + 1]]
            assert len(set(toks.tolist())) == len(toks) and np.all(np.diff(toks) > 0)
