/*
 * gptq.h -- C ABI of the GB300 (sm_103a) GPTQ mixed-precision GEMM library.
 *
 * The library multiplies fp16/bf16 activations by 2/3/4/8-bit GPTQ weights packed in int32
 * words, dequantizing group-wise with  w = (q - zero) * scale.  It follows the page
 * "增强 vLLM 对 GPTQv2 格式的支持：分析与实现" (xxxxyu.github.io):
 *   section "LLM 的权重量化"             quantizer, its inverse w_hat = (q - zero) * scale,
 *                                        symmetric zero round((2^b - 1) / 2);
 *   section "从 GPTQv1 到 GPTQv2"         v1 checkpoints store clamp(zero - 1) and add 1 at run
 *                                        time, v2 checkpoints store zero; v1 -> v2 is lossless;
 *   section "调整细节：根据格式选择处理方式" the gptq_gemm op takes a use_v2_format flag and
 *                                        adds zero_offset = use_v2_format ? 0 : 1 to the
 *                                        unpacked zeros.
 *
 * Layouts (all row-major, contiguous, no padding between rows):
 *   A        [M, K]             fp16 or bf16 activations (a_dtype)
 *   qweight  [K * bits / 32, N] int32; column n is an LSB-first bit stream of its K codes:
 *                               code k occupies stream bits [bits*k, bits*k + bits), the
 *                               stream's words being qweight[0][n], qweight[1][n], ...
 *                               (2/4/8-bit: 16/8/4 codes per word; 3-bit: 32 codes in
 *                               every 3 consecutive words, two codes straddling words)
 *   qzeros   [G, N * bits / 32] int32; row g is an LSB-first stream of the N stored zeros
 *   scales   [G, N]             fp16
 *   g_idx    [K]                int32 group of each input row (act-order), or NULL
 *   C        [M, N]             same dtype as A
 *   W        [K, N]             dequantized weights (fp16 or bf16)
 * where G = K / group, or G = 1 when group == -1 (one group spanning all rows).
 * Words are bit patterns (read as uint32).  The runtime zero is stored + 1 for
 * GPTQ_FMT_V1 and stored for GPTQ_FMT_V2, in plain integer arithmetic.
 *
 * Shapes the library accepts: K > 0 and N > 0, both multiples of 32; group == -1 or a
 * positive divisor of K; g_idx only with group != -1, every entry in [0, G).  M >= 0;
 * M == 0 is a no-op.
 *
 * Ownership: the caller allocates and frees every buffer.  Device entry points take device
 * pointers, must be 16-byte aligned (g_idx: 4-byte), and run asynchronously on `stream`
 * (a cudaStream_t; NULL = legacy default stream) on the current device.  The library keeps
 * only a per-device status word and per-device launch attributes; it never allocates device
 * memory in these calls.  gptq_gemm_host is the exception: it takes A and C in host memory and
 * returns only once the stream has drained.
 *
 * Stream order: the GEMM entry points (gptq_gemm, gptq_gemm_perm, gptq_gemm_perm_noalloc) use
 * programmatic dependent launch, so their kernels may start while the kernel issued just before
 * them on `stream` is still running.  They read A (and perm) only after that kernel has
 * completed, but they may read the checkpoint -- qweight, qzeros, scales, g_idx -- before, to
 * start the weight stream early.  Hence the checkpoint must not be written by the kernel issued
 * immediately before the call on the same stream (nor by a kernel still running when that one
 * starts, which only a caller that itself uses programmatic dependent launch can arrange).  A
 * checkpoint written by gptq_quantize_rtn may be used by the very next call: that entry point
 * ends with an ordering step of its own.  gptq_gemm_grouped reads everything after the wait.
 *
 * Errors: every entry point returns GPTQ_OK (0) or a negative gptq_status from host-side
 * validation or a failed launch; nothing is launched when validation fails.  Kernels never
 * trap: a bounded wait that runs out, or an act-order index outside [0, G), sets a bit in
 * the device status word, read and cleared by gptq_get_device_status().
 */
#ifndef GPTQ_GB300_H
#define GPTQ_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { GPTQ_FMT_V1 = 1, GPTQ_FMT_V2 = 2 } gptq_fmt;
typedef enum { GPTQ_F16 = 0, GPTQ_BF16 = 1 } gptq_dtype;

typedef enum {
  GPTQ_OK = 0,
  GPTQ_ERR_ARG = -1,            /* NULL required pointer, bits/fmt/dtype/sym out of range */
  GPTQ_ERR_SHAPE = -2,          /* K/N not multiples of 32, group does not divide K, g_idx
                                   with group == -1, negative M, too many groups           */
  GPTQ_ERR_ALIGN = -3,          /* a pointer not 16-byte aligned (g_idx: 4-byte)            */
  GPTQ_ERR_WORKSPACE = -4,      /* workspace smaller than gptq_gemm_workspace_size()        */
  GPTQ_ERR_ZERO_OVERFLOW = -5,  /* v1 -> v2 repack of a stored zero equal to 2^bits - 1     */
  GPTQ_ERR_CUDA = -6,           /* a CUDA runtime call or launch failed                     */
  GPTQ_ERR_UNSUPPORTED = -7,    /* the current device is not a Blackwell sm_10x part        */
  GPTQ_ERR_DEVICE = -8          /* the device status word reported an error                 */
} gptq_status;

/* Bits of the device status word (see gptq_get_device_status). */
#define GPTQ_DEV_TIMEOUT 0x1u     /* a bounded wait inside a kernel ran out; output invalid */
#define GPTQ_DEV_GIDX_RANGE 0x2u  /* an act-order g_idx entry was outside [0, G)            */
#define GPTQ_DEV_SCALE_OVERFLOW 0x4u /* gptq_quantize_rtn: a group's scale overflowed fp16   */
#define GPTQ_DEV_EXPERT_ROWS 0x8u /* gptq_gemm_grouped: an expert's row range was decreasing,
                                     outside [0, rows] or longer than max_m; its rows of C
                                     were not written                                        */
#define GPTQ_DEV_GIDX_GROUPS 0x10u /* gptq_prepack_act_order_device: g_idx had an entry outside
                                     [0, K/group) or a group not of exactly `group` rows;
                                     qweight_out and perm were not written                   */

/*
 * gptq_dequant -- write the dequantized weights W[k][n] = RN((q - zero) * scale).
 * Page section "LLM 的权重量化" (w_hat = (q - zero) * scale) and the reconstruct kernel in
 * "调整细节：根据格式选择处理方式" (zeros[i] + zero_offset).  The product is taken in fp32,
 * where it is exact, and rounded once, to nearest-even, to out_dtype, so W is bit-exact.
 * Device pointers: qweight, qzeros, scales, g_idx (nullable), W_out [K, N].
 * Returns GPTQ_OK or a negative gptq_status.  An out-of-range g_idx entry is clamped to
 * [0, G) and flagged with GPTQ_DEV_GIDX_RANGE.
 */
int gptq_dequant(const int32_t* qweight, const int32_t* qzeros, const void* scales,
                 const int32_t* g_idx, int K, int N, int bits, int group, int fmt,
                 int out_dtype, void* W_out, void* stream);

/*
 * gptq_gemm -- C[M, N] = A[M, K] @ W[K, N] with W dequantized on the fly, the operation
 * vLLM's gptq_gemm(..., use_v2_format) performs (page section "调整细节：根据格式选择处理
 * 方式"; fmt == GPTQ_FMT_V2 is use_v2_format = true).  Products are accumulated in fp32 and
 * C is rounded once to A's dtype.  M <= 32 runs the memory-bound decode kernel (TMA-streamed
 * weights, mma.sync from registers, split-K over a thread-block cluster reduced through
 * distributed shared memory); larger M runs the tcgen05 tensor-core kernel, and so does M <= 32
 * when K is so long that the decode kernel's staged activations fit no CTA even split 16 ways
 * (K beyond 28672 with many tokens).
 * The multiply is fp16 x fp16 with fp32 accumulation for both activation types: weights are
 * rounded once to fp16 (the exact product (q - zero) * scale, as gptq_dequant gives it), and
 * bf16 activations are multiplied as fp16 times a power of two per row (exact for every value
 * in fp16's normal range; values more than 2^29 below the row's largest may round), the power
 * of two multiplied back into the fp32 result.  A weight rounded to bf16 would carry up to 2^-8
 * relative error, more than the 2e-3 accuracy bound; fp16 carries 2^-11.  Consequently a
 * dequantized weight beyond fp16's range (|(q - zero) * scale| > 65504, i.e. scale > 256 for
 * 8-bit codes) is outside what the per-weight and tensor-core paths handle, for either dtype.
 * Device pointers: A, qweight, qzeros, scales, g_idx (nullable), C, workspace.  `workspace`
 * (16-byte aligned, owned by the caller) is used only when A is bf16 and the tensor-core kernel
 * runs: it then holds the fp16 copy of A and its row scales and must be at least
 * gptq_gemm_workspace_size() bytes (GPTQ_ERR_WORKSPACE otherwise, nothing launched).  With fp16
 * activations, or M <= 32 and K within the decode kernel's reach, it may be NULL.
 * Act-order (g_idx given): with a workspace of at least
 * gptq_gemm_act_order_workspace_size(M, K, N, bits, group) bytes (nonzero), the call sorts the
 * rows by group on the device (the stable sort of gptq_prepack_act_order), writes the sorted
 * packed weight into the workspace and runs the group-wise kernels on it with A's columns taken
 * through the sort -- the same result as gptq_prepack_act_order + gptq_gemm_perm, computed per
 * call.  When g_idx does not describe groups of exactly `group` rows (or holds an entry outside
 * [0, G)), a device flag routes the call to the per-row-group kernels instead, inside the same
 * launches' stream order, with no host synchronisation.  A smaller workspace selects those
 * per-row-group kernels directly.
 * Returns GPTQ_OK or a negative gptq_status.
 */
int gptq_gemm(const void* A, int M, int K, int a_dtype, const int32_t* qweight,
              const int32_t* qzeros, const void* scales, const int32_t* g_idx, int N, int bits,
              int group, int fmt, void* C, void* workspace, size_t workspace_bytes,
              void* stream);

/*
 * gptq_gemm_host -- gptq_gemm with the activations and the result in host memory: copies
 * A_host [M, K] (16-bit, a_dtype) into the device buffer A_dev, runs gptq_gemm on `stream` with
 * C in the device buffer C_dev, copies C_dev [M, N] into C_host and waits for the stream, so
 * that C_host holds the result when the call returns.  The operation is gptq_gemm's (page
 * section "调整细节：根据格式选择处理方式"); every other argument means what it means there.
 * Host pointers: A_host, C_host.  Page-locked memory that the device reaches at the same
 * address is read and written by kernels over the chip-to-chip link: A is copied into A_dev by a
 * kernel that the GEMM overlaps, and when the decode kernels take the problem (M <= 32, no
 * g_idx) they write C straight into C_host, leaving C_dev untouched.  Pageable memory works,
 * through DMA copies.  Device pointers: A_dev (M*K*2 bytes), C_dev (M*N*2
 * bytes), qweight, qzeros, scales, g_idx (nullable), workspace; all owned by the caller.
 * Returns GPTQ_OK, GPTQ_ERR_ARG for a NULL host or staging pointer, any gptq_gemm status, or
 * GPTQ_ERR_CUDA if a copy or the synchronisation failed.  gptq_gemm's argument checks run
 * before anything is copied; a status found when the kernels are chosen (GPTQ_ERR_WORKSPACE for
 * a bf16 problem that the tensor-core kernel takes) comes after the copy of A, with the stream
 * drained and C_host not written.  M == 0 returns GPTQ_OK with nothing copied.
 */
int gptq_gemm_host(const void* A_host, void* A_dev, int M, int K, int a_dtype,
                   const int32_t* qweight, const int32_t* qzeros, const void* scales,
                   const int32_t* g_idx, int N, int bits, int group, int fmt, void* C_dev,
                   void* C_host, void* workspace, size_t workspace_bytes, void* stream);

/*
 * gptq_host_plan_create / _run / _destroy -- gptq_gemm_host prepared once for a loop that reruns
 * one problem on the same buffers (only the contents of A_host change between runs): create
 * makes one gptq_gemm_host call (which checks everything and returns its status) and then
 * captures the stream work of such a call into a CUDA graph; each run replays it on `stream` --
 * A_host's current contents in, the GEMM, the result in C_host -- and returns once the stream
 * has drained.  Arguments as for gptq_gemm_host; `stream` must not be NULL (the legacy default
 * stream cannot be captured: GPTQ_ERR_ARG).  The buffers must outlive the plan.  create returns
 * GPTQ_OK with *plan set, or an error status with *plan NULL; run returns GPTQ_OK, GPTQ_ERR_ARG
 * for a NULL plan, or GPTQ_ERR_CUDA; destroy (NULL allowed) returns GPTQ_OK.
 */
typedef struct gptq_host_plan gptq_host_plan;
int gptq_host_plan_create(gptq_host_plan** plan, const void* A_host, void* A_dev, int M, int K,
                          int a_dtype, const int32_t* qweight, const int32_t* qzeros,
                          const void* scales, const int32_t* g_idx, int N, int bits, int group,
                          int fmt, void* C_dev, void* C_host, void* workspace, size_t workspace_bytes,
                          void* stream);
int gptq_host_plan_run(gptq_host_plan* plan);
int gptq_host_plan_destroy(gptq_host_plan* plan);

/*
 * gptq_prepack_act_order -- HOST function: rewrite an act-order checkpoint (page section
 * "LLM 的权重量化": the quantization groups are the row sets {k : g_idx[k] == g}) so that the
 * groups are contiguous row ranges.  perm[k'] (the stable sort of the rows by g_idx) is the
 * original row now at row k'; qweight_out holds W[perm[k'], n] in the layout above, so rows
 * [g*group, (g+1)*group) belong to group g and qzeros/scales stay valid unchanged.  Then
 * A @ W == A[:, perm] @ W_out: gptq_gemm_perm computes it, gathering A through perm.
 * Host memory: qweight [K*bits/32, N], g_idx [K], qweight_out (same size, must not alias
 * qweight), perm [K].  Every group must hold exactly `group` rows (as GPTQ's act-order does),
 * else GPTQ_ERR_SHAPE; an entry outside [0, K/group) is GPTQ_ERR_SHAPE too.
 */
int gptq_prepack_act_order(const int32_t* qweight, const int32_t* g_idx, int K, int N, int bits,
                           int group, int32_t* qweight_out, int32_t* perm);

/*
 * gptq_prepack_act_order_device -- gptq_prepack_act_order for a checkpoint already in device
 * memory, asynchronously on `stream` (page section "LLM 的权重量化": the groups are the row sets
 * {k : g_idx[k] == g}).  It runs the stable sort and the repack that gptq_gemm's act-order path
 * runs on every call, once: a model's load step, after which gptq_gemm_perm multiplies the
 * sorted copy on every call.  perm and qweight_out are bit-identical to the host function's.
 * Device pointers: qweight [K*bits/32, N], g_idx [K], qweight_out (same size as qweight, must not
 * overlap it), perm [K], workspace (at least gptq_prepack_act_order_device_workspace_size(K, bits,
 * group) bytes, caller-owned, overwritten).  Alignment: 16 bytes for qweight, qweight_out, perm
 * and workspace; 4 for g_idx.
 * Returns GPTQ_OK or a negative gptq_status (GPTQ_ERR_SHAPE where the workspace size is 0,
 * GPTQ_ERR_WORKSPACE, GPTQ_ERR_ARG for overlapping weights); nothing is launched then.  A g_idx
 * with an entry outside [0, K/group), or a group that does not hold exactly `group` rows, is found
 * on the device: qweight_out and perm are left unwritten and GPTQ_DEV_GIDX_GROUPS is set in the
 * device status word.  The call ends with an ordering step, so a GEMM may use qweight_out and
 * perm as the very next call on the stream.
 */
int gptq_prepack_act_order_device(const int32_t* qweight, const int32_t* g_idx, int K, int N, int bits,
                                  int group, int32_t* qweight_out, int32_t* perm, void* workspace,
                                  size_t workspace_bytes, void* stream);

/* Bytes of device workspace gptq_prepack_act_order_device needs: 256 + K * 4 rounded up to 256.
 * 0 when the device sort does not take the shape (bits not 2/3/4/8, K not a multiple of 32 or of
 * group, G * 128 + K * 2 above 200 KB, a group of more than 65535 rows, or a packed column of
 * more than 200 KB in 4-column strips); the host function remains for those. */
size_t gptq_prepack_act_order_device_workspace_size(int K, int bits, int group);

/*
 * gptq_gemm_perm -- C[M, N] = A[:, perm] @ W[K, N] for a checkpoint prepacked by
 * gptq_prepack_act_order (W = its qweight_out, contiguous groups of `group` rows), i.e. the
 * act-order GEMM of page section "调整细节：根据格式选择处理方式" without a per-row group
 * lookup.  One token: the decode kernel gathers A's columns through perm while staging them.
 * Several tokens: A[:, perm] is first gathered once into `workspace` (a device buffer of at least
 * gptq_gemm_perm_workspace_size(M, K) bytes, 16-byte aligned, owned by the caller; it is
 * overwritten), then the decode kernel reads it.  Tokens: 0 <= M <= 32 (larger M:
 * GPTQ_ERR_SHAPE; gptq_gemm with g_idx serves that range).
 * Device pointers: A [M, K], perm [K] int32 (16-byte aligned; an entry outside [0, K) is
 * clamped, never read past A), qweight, qzeros, scales, C, workspace.
 * Returns GPTQ_OK or a negative gptq_status (GPTQ_ERR_WORKSPACE if the workspace is too small;
 * GPTQ_ERR_SHAPE, with nothing computed, if K is so long that the decode kernel's staged
 * activations for M tokens fit no CTA even split 16 ways, which only K beyond 28672 reaches).
 */
int gptq_gemm_perm(const void* A, int M, int K, int a_dtype, const int32_t* perm,
                   const int32_t* qweight, const int32_t* qzeros, const void* scales, int N,
                   int bits, int group, int fmt, void* C, void* workspace,
                   size_t workspace_bytes, void* stream);

/* Bytes of workspace gptq_gemm_perm needs: M * K * 2 rounded up to 256 for M > 1, else 0. */
size_t gptq_gemm_perm_workspace_size(int M, int K);

/*
 * gptq_gemm_grouped -- the quantized mixture-of-experts GEMM: for every expert e in [0, E),
 * C[r, :] = A[r, :] @ W_e for the rows r in [offsets[e], offsets[e + 1]), with W_e expert e's
 * GPTQ weight dequantized on the fly exactly as in gptq_gemm.  Page "4.3 Weight-only INT4 量化：
 * GPTQ、AWQ 与 Marlin Kernel", section 7 ("vLLM 生态：GPTQ/AWQ 的工程现状"): GPTQ checkpoints of
 * MoE models quantize every expert's weights, and vLLM runs them through a fused MoE path.  The
 * pages fix no layout; the one here is the plainest: the rows of A are already grouped by expert
 * (the caller gathers and orders them), and every expert has the same K, N, bits and group.
 * One launch covers all experts (one decode kernel with min(E, rows) expert slots as its third
 * grid dimension: no more experts than rows can hold rows, and each slot takes the next expert
 * that does).
 * Device pointers:
 *   A        [rows, K] fp16/bf16 (a_dtype), 16-byte aligned;
 *   offsets  [E + 1] int32, nondecreasing, offsets[0] = 0, offsets[E] <= rows, 4-byte aligned;
 *            read on the device after the previous kernel on the stream has finished, so a
 *            routing kernel may write them just before;
 *   qweight  [E][K * bits / 32][N], qzeros [E][G][N * bits / 32], scales [E][G][N] fp16
 *            (each expert's tensors laid out as for gptq_gemm, experts back to back);
 *   C        [rows, N] of a_dtype; rows outside every expert's range are left untouched.
 * max_m (1..32) bounds every expert's row count; it selects the kernel's token tile.  An expert
 * whose range is decreasing, leaves [0, rows] or exceeds max_m is skipped and flagged with
 * GPTQ_DEV_EXPERT_ROWS.  No g_idx (act-order experts: prepack them, one gptq_gemm_perm each).
 * Returns GPTQ_OK (also for rows == 0 or E == 0, with no launch) or a negative gptq_status
 * (GPTQ_ERR_SHAPE, with nothing launched, if K is so long that max_m tokens' staged activations
 * fit no CTA even split 16 ways: K beyond 28672).
 */
int gptq_gemm_grouped(const void* A, int rows, int K, int a_dtype, const int32_t* offsets, int E,
                      int max_m, const int32_t* qweight, const int32_t* qzeros, const void* scales,
                      int N, int bits, int group, int fmt, void* C, void* stream);

/*
 * gptq_gemm_perm_noalloc -- gptq_gemm_perm for callers that cannot allocate device memory: a
 * serving runtime or framework plug-in whose allocator has reserved the GPU's memory up front
 * and forbids further allocations, or code for which the synchronisation of cudaMalloc is not
 * allowed.  Same arguments and result as gptq_gemm_perm, without the workspace: the gathered
 * activations live in a static device buffer of 1 MiB that every GPU loading this library holds
 * until the process exits.  Limit: M * K * 2 bytes <= 1 MiB (e.g. M = 32 with K <= 16384);
 * larger problems return GPTQ_ERR_WORKSPACE.  The call allocates nothing (no cudaMalloc or
 * cudaFree, no allocating library routine).  The first call on a device looks up the buffer's
 * device address there (cudaGetSymbolAddress); make that first call before any stream capture.
 * All calls share the buffer and leave their contents in it (each call writes every element it
 * later reads): calls that overlap on the GPU, on any streams, race.  The pages have no
 * counterpart for this entry point.
 */
int gptq_gemm_perm_noalloc(const void* A, int M, int K, int a_dtype, const int32_t* perm,
                           const int32_t* qweight, const int32_t* qzeros, const void* scales,
                           int N, int bits, int group, int fmt, void* C, void* stream);

/*
 * gptq_prepack_interleave -- HOST function: rewrite qweight into the decode kernel's own layout,
 * the offline reordering the page "4.3 Weight-only INT4 量化：GPTQ、AWQ 与 Marlin Kernel" (section
 * 6.1) describes for Marlin: packed words arranged so that what one lane of the kernel loads is
 * contiguous.  The codes, their packing inside a word and qzeros / scales are unchanged; only
 * whole words move.  Every 32-column block becomes one contiguous run along K; inside it each
 * k-tile (4 units: 32/bits * 4 consecutive k, 128 for 3-bit) is 512 bytes per qweight row of a
 * unit, in lane order: word (((cb * T + kt) * R + r) * 32 + lane) * 4 + c holds checkpoint row
 * (4 kt + t) * R + r and column 32 cb + 4 q + c, where lane = 4 g + t, q = (g & 1) * 4 + g / 2,
 * T = K * bits / 128 (K / 128 for 3-bit) k-tiles and R = 3 rows per unit for 3-bit, else 1.
 * A warp's 16-byte fragment loads then read 512 contiguous bytes (no swizzle), and the kernel
 * copies each warp's part of a chunk with one 1D bulk copy (no tensor map).
 * qweight, qweight_il: host arrays of K * bits / 32 * N int32 (they may not overlap).
 * Shapes: N a multiple of 32, K a multiple of 4 * 32 / bits (128 for 3-bit).
 * Returns GPTQ_OK, GPTQ_ERR_ARG or GPTQ_ERR_SHAPE.
 */
int gptq_prepack_interleave(const int32_t* qweight, int K, int N, int bits, int32_t* qweight_il);

/*
 * gptq_gemm_interleaved -- gptq_gemm (M <= 32, the decode kernel) on a checkpoint whose qweight
 * went through gptq_prepack_interleave; qzeros and scales are the checkpoint's own.  `perm`
 * (nullable) is the act-order permutation of gptq_prepack_act_order, for a checkpoint sorted by
 * group before it was interleaved; then C = A[:, perm] @ W and, for M > 1, `workspace` takes
 * gptq_gemm_perm_workspace_size(M, K) bytes (otherwise it may be NULL).  The groups must be whole
 * k-tiles (group a multiple of 4 * 32 / bits, 128 for 3-bit; -1 allowed): the scale folds per
 * group.  Same arithmetic, results and stream-order rules as gptq_gemm.
 * Returns GPTQ_OK or a negative gptq_status (GPTQ_ERR_SHAPE for M > 32 or misaligned K/group).
 */
int gptq_gemm_interleaved(const void* A, int M, int K, int a_dtype, const int32_t* perm,
                          const int32_t* qweight_il, const int32_t* qzeros, const void* scales, int N,
                          int bits, int group, int fmt, void* C, void* workspace, size_t workspace_bytes,
                          void* stream);

/* Bytes of device workspace gptq_gemm may need for this problem: the fp16 copy of bf16
 * activations and their row scales, (M * K * 2 rounded up to 256) + (M * 4 rounded up to 256);
 * 0 for M <= 0.  Enough for every activation dtype and path. */
size_t gptq_gemm_workspace_size(int M, int K, int N, int bits, int group);

/* Bytes of device workspace with which gptq_gemm runs an act-order problem (g_idx given) on
 * rows sorted by group on the device: a flag (256 bytes), the sorted row order and each sorted
 * row's code position (K * 4 bytes each, rounded up to 256), the sorted packed weight
 * (K * bits / 32 * N * 4, rounded up to 256) and gptq_gemm_workspace_size(max(M, 1), K, ...).
 * 0 when the shape does not qualify: K % group, G * 128 + K * 2 above 200 KB (the sort's shared
 * memory), a group of more than 65535 rows, a packed column of more than 200 KB in 4-column
 * strips, or a group size that is not a multiple of 4 * (32 / bits) rows (128 rows for 3-bit);
 * gptq_gemm then always uses the per-row-group kernels. */
size_t gptq_gemm_act_order_workspace_size(int M, int K, int N, int bits, int group);

/*
 * gptq_repack_zeros_v1_to_v2 -- HOST function: rewrite a v1 qzeros array ([G, N*bits/32],
 * host memory) as v2 by adding 1 to every stored field (page section "从 GPTQv1 到 GPTQv2":
 * the conversion is lossless).  A v1 field of 2^bits - 1 has no v2 encoding: the call then
 * returns GPTQ_ERR_ZERO_OVERFLOW and leaves qz_v2 unchanged.  qz_v1 and qz_v2 may alias.
 */
int gptq_repack_zeros_v1_to_v2(const int32_t* qz_v1, int32_t* qz_v2, int G, int N, int bits);

/*
 * gptq_quantize_rtn -- write a GPTQ checkpoint from fp32 weights on the device with the
 * page's round-to-nearest quantizer (section "LLM 的权重量化"):
 *   asymmetric: scale = (wmax - wmin) / (2^b - 1), zero = clamp(-round(wmin / scale)),
 *   symmetric:  scale = 2 max|w| / (2^b - 1),      zero = round((2^b - 1) / 2),
 *   q = clamp(round(w / scale) + zero, 0, 2^b - 1),
 * over each group of rows (rows k with g_idx[k] == g when g_idx is given).  The scale is
 * computed in fp32 and stored as fp16; zero and q use the stored scale; round is
 * half-to-even; a scale that rounds to 0 is stored as 1.  fmt == GPTQ_FMT_V1 stores
 * clamp(zero - 1) (section "从 GPTQv1 到 GPTQv2").
 * Device pointers: W [K, N] fp32, g_idx (nullable), qweight, qzeros, scales (outputs).
 * Returns GPTQ_OK or a negative gptq_status.
 */
int gptq_quantize_rtn(const float* W, int K, int N, int bits, int group, const int32_t* g_idx,
                      int sym, int fmt, int32_t* qweight, int32_t* qzeros, void* scales,
                      void* stream);

/*
 * gptq_get_device_status -- synchronize `stream`, then read and clear the current device's
 * status word (GPTQ_DEV_* bits; 0 = no error since the last call).  Returns GPTQ_OK, or
 * GPTQ_ERR_CUDA if the synchronize or the read failed.
 */
int gptq_get_device_status(void* stream, unsigned int* out);

/*
 * gptq_selftest_wait_timeout -- exercise the failure path of the kernels' bounded waits without
 * faulting the GPU: one CTA waits, with the same wait routine the tensor-core kernel uses, on an
 * mbarrier phase that nothing completes.  After `limit_ns` (1 ns .. 10 s) the wait gives up,
 * sets GPTQ_DEV_TIMEOUT in the device status word and writes 1 to *waited_out (a device int,
 * 4-byte aligned); the kernel then returns and the context stays usable.  Read the status with
 * gptq_get_device_status().  No counterpart on the pages: this is the library's own test hook.
 */
int gptq_selftest_wait_timeout(unsigned long long limit_ns, int* waited_out, void* stream);

/* Human-readable name of a gptq_status code (static string). */
const char* gptq_strerror(int code);

#ifdef __cplusplus
}
#endif

#endif /* GPTQ_GB300_H */
