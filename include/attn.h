/*
 * attn.h -- C ABI of libattn_gb300.so, the GB300 (sm_103a) multi-head
 * attention forward.
 *
 * The operation is O = softmax(scale · Q·K^T) · V per (batch, head), taken
 * from "Transformer算子生态深度分析" chapter 2 (自注意力机制算子): scores in
 * §2.2, row-wise softmax in §2.3, weighted sum in §2.4.  attn_fwd computes it
 * tile by tile with the online-softmax merge of §2.6 (running max m and
 * running exp-sum, previous output rescaled by exp(m_old - m)), so the S×S
 * score and probability matrices never reach device memory.
 *
 * Conventions shared by every entry point
 * ----------------------------------------
 *  - All tensor pointers are DEVICE pointers owned by the caller.  The
 *    library keeps no reference to them after the call is enqueued and
 *    allocates no device memory of its own (it holds one 4-byte status word
 *    per device and the fixed scratch of qkv_proj_attn_noalloc, both
 *    statically declared device variables).
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *    default stream).  None of them synchronises, except
 *    attn_get_device_status.
 *  - Element types (`dtype`): ATTN_F32, ATTN_F16, ATTN_BF16.  q, k, v, o
 *    share one dtype.  16-bit inputs are multiplied on the tensor cores with
 *    fp32 accumulation; softmax statistics are fp32 (the mixed-precision
 *    split of "WebGPU 算子优化：QKV 内存合并与 FlashAttention 分块计算",
 *    §浏览器端落地的关键参数与监控).  ATTN_F32 runs exact fp32 FMA arithmetic.
 *  - Layouts (`layout`), from the same WebGPU page, §QKV 矩阵的内存合并模式选择:
 *      ATTN_LAYOUT_BHSD  contiguous        [B, h, S, d]
 *      ATTN_LAYOUT_BSHD  head-interleaved  [B, S, h, d]
 *    q, k, v and o all use the given layout, densely packed.
 *  - lse (optional, may be NULL) is fp32 [B, h, S]: the natural-log
 *    log-sum-exp of each query row's scaled scores, in both layouts.
 *  - `scale` <= 0 selects the default 1/sqrt(d) ("Transformer算子生态深度分析"
 *    §2.2, variance argument).
 *  - Return value: ATTN_OK (0) when the work was enqueued; a negative
 *    ATTN_E_* code when an argument is invalid, in which case nothing was
 *    launched and no CUDA call was made; a positive value is a cudaError_t
 *    reported by the runtime while enqueuing.
 *  - Device-side faults of the pipeline (a wait that exceeded its time
 *    limit) do not trap: the kernel records a code in the device status
 *    word and returns; read it with attn_get_device_status.  There is one
 *    status word per device, shared by every stream: once a timeout is
 *    recorded, every attention kernel launched afterwards on that device, on
 *    any stream, does no work (its output is left undefined) until
 *    attn_get_device_status has read and cleared the word.  Callers that use
 *    several streams should check the status after each batch of work.
 */
#ifndef ATTN_GB300_H
#define ATTN_GB300_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { ATTN_LAYOUT_BHSD = 0, ATTN_LAYOUT_BSHD = 1, ATTN_LAYOUT_GROUPED = 2 } attn_layout;
typedef enum { ATTN_F32 = 0, ATTN_F16 = 1, ATTN_BF16 = 2 } attn_dtype;

enum {
  ATTN_OK = 0,
  ATTN_E_NULL = -1,      /* a required pointer is NULL                                 */
  ATTN_E_SHAPE = -2,     /* B, h, S < 1; d unsupported for the dtype; D != h*d; too large */
  ATTN_E_ALIGN = -3,     /* a tensor pointer is not 16-byte aligned                    */
  ATTN_E_LAYOUT = -4,    /* layout is not ATTN_LAYOUT_BHSD / ATTN_LAYOUT_BSHD          */
  ATTN_E_DTYPE = -5,     /* dtype unknown, or not supported by this entry point        */
  ATTN_E_WORKSPACE = -6, /* workspace NULL, misaligned or smaller than required        */
  ATTN_E_ALIAS = -7,     /* the output overlaps an input or the workspace              */
  ATTN_E_DEVICE = -8,    /* no usable sm_103 device / driver entry point missing       */
  ATTN_E_TIMEOUT = -9,   /* (device status only) a pipeline wait exceeded its limit    */
  ATTN_E_SCRATCH_LIMIT = -10, /* problem too large for qkv_proj_attn_noalloc's fixed scratch */
  ATTN_E_MISMATCH = -11  /* attn_compare: the two outputs differ by more than atol     */
};

typedef enum { ATTN_KERNEL_NAIVE = 0, ATTN_KERNEL_ONLINE = 1 } attn_kernel;

/*
 * attn_fwd -- fused attention forward (online softmax, one kernel launch).
 *
 *   q, k, v  [in]  B·h·S·d elements each, in `layout`, of `dtype`.
 *   o        [out] same shape, layout and dtype as q.  Must not overlap q, k, v.
 *   lse      [out] optional fp32 [B, h, S]; NULL to skip.
 *   B, h, S, d     batch, heads, sequence length, head dimension.
 *                  16-bit dtypes: d in {64, 128}.  ATTN_F32: 1 <= d <= 256.
 *   scale          softmax scale; <= 0 means 1/sqrt(d).
 *   layout, dtype  see above.
 *   stream         cudaStream_t to enqueue on.
 *
 * Non-causal: every query attends to all S keys.  All pointers must be
 * 16-byte aligned.  Errors: ATTN_E_NULL, ATTN_E_SHAPE, ATTN_E_ALIGN,
 * ATTN_E_LAYOUT, ATTN_E_DTYPE, ATTN_E_ALIAS, ATTN_E_DEVICE, or a cudaError_t.
 *
 * Kernels: 16-bit problems stream K and V through a pipelined kernel; for
 * d = 64 and S <= 512, when the head count leaves it no more waves of work
 * than the streaming kernel, one CTA per (batch, head) keeps the head's Q, K
 * and V resident in shared memory instead (no per-item pipeline start and
 * drain).  Both compute the same result up to fp32 summation order.  The
 * environment variable ATTN_RESIDENT=never|force overrides the choice (for
 * tests and comparisons).
 */
int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int h, int S,
             int d, float scale, int layout, int dtype, void* stream);

/*
 * attn_fwd_ws -- attn_fwd with a caller scratch buffer that lets the kernel
 * balance the last wave.  The work items are (batch, head, 256 query rows);
 * attn_fwd deals whole items to at most one CTA per SM, so when the item
 * count is not a multiple of the SM count the last wave leaves SMs idle.
 * With the scratch, the last one to two waves of items are cut along the key
 * axis into equal runs of 128-key tiles, one run per SM (see
 * attn_flash_schedule).  Each later piece of
 * a cut item leaves its running max m, exp-sum l and unnormalised output in
 * the scratch; the piece that starts at key 0 merges them into its own with
 * the merge rule of "Transformer算子生态深度分析" §2.6 (each side rescaled by
 * exp(m_side - m), then added), the rule that also merges consecutive key
 * tiles.  The result equals attn_fwd's up to fp32 rounding order.
 *
 *   workspace  [in/out] device scratch of at least
 *              attn_fwd_ws_bytes(B, h, S, d, dtype) bytes, 256-byte aligned,
 *              owned by the caller and used by this call until the stream
 *              reaches it; its contents on entry do not matter.  NULL with
 *              ws_bytes = 0 runs attn_fwd.
 *   other arguments, lse and layouts as attn_fwd.  ATTN_F32 ignores the
 *   workspace (the fp32 path has no waves to balance).
 *
 * Items are cut only where it pays: at d = 64, when they have at least 16
 * key tiles and the cut saves at least 8 key-tile steps per SM (otherwise
 * attn_fwd_ws runs as attn_fwd and attn_fwd_ws_bytes reports 0).  The
 * environment variable ATTN_SPLIT=never disables the cut and ATTN_SPLIT=force
 * cuts whenever the item count leaves a partial wave (for tests).
 *
 * Errors: as attn_fwd, plus ATTN_E_WORKSPACE (misaligned, or smaller than
 * attn_fwd_ws_bytes for the current device) and ATTN_E_ALIAS (workspace
 * overlaps a tensor).
 */
int attn_fwd_ws(const void* q, const void* k, const void* v, void* o, float* lse, int B, int h,
                int S, int d, float scale, int layout, int dtype, void* workspace, size_t ws_bytes,
                void* stream);

/*
 * The work schedule attn_fwd_ws (split = 1) or attn_fwd (split = 0) would
 * use for a 16-bit problem on a GPU with num_sms SMs.  Host only: no device is
 * needed and nothing is launched.  Outputs (each may be NULL):
 *   mode      0: one item per CTA (d = 128); 1: whole items on a persistent
 *             grid, item i on CTA i mod grid; 2: as 1 for items [0, dp_end),
 *             then the sk_units key tiles of the remaining items cut into
 *             runs, CTA g taking tiles [cut[g], cut[g+1]) in item-major order
 *   grid      CTAs launched
 *   dp_end, sk_units   as above (sk_units = 0 unless mode = 2)
 *   cut       [grid + 1] run bounds, written only in mode 2 (grid <= 256)
 *   g_last    [grid], mode 2 only: the CTA whose run holds the last key tile
 *             of the item in which CTA g's run ends
 * An item is (batch, head, 256 query rows) with ceil(S / 128) key tiles.
 * Honours ATTN_SPLIT like attn_fwd_ws.  Returns 0, or ATTN_E_SHAPE (B, h, S or
 * num_sms < 1, d not 64 or 128).
 */
int attn_flash_schedule(int B, int h, int S, int d, int num_sms, int split, int* mode, int* grid,
                        long long* dp_end, long long* sk_units, long long* cut, int* g_last);

/*
 * Scratch bytes attn_fwd_ws needs on the current device (it depends on the
 * SM count): per SM 64 bytes of flags and 256 rows of (m, l) and d fp32
 * values.  0 when no item would be cut (see above: d = 128, short items, an
 * item count that fills whole waves), for ATTN_F32, for unsupported sizes, or
 * without a device.
 */
size_t attn_fwd_ws_bytes(int B, int h, int S, int d, int dtype);

/*
 * attn_fwd_mixed -- fp32 inputs, 16-bit output: the mixed-precision split of
 * "WebGPU 算子优化：QKV 内存合并与 FlashAttention 分块计算",
 * §浏览器端落地的关键参数与监控 (16-bit score products, fp32 softmax
 * statistics, 16-bit output) for callers that hold Q, K, V in fp32.
 *
 *   q, k, v    [in]  fp32, B·h·S·d elements each, in `layout`.
 *   o          [out] `out_dtype` (ATTN_F16 or ATTN_BF16), same shape and layout.
 *   lse        [out] optional fp32 [B, h, S].
 *   workspace  device scratch, 256-byte aligned, of
 *              attn_fwd_mixed_workspace_bytes(B, h, S, d, out_dtype) bytes or
 *              more; exactly 3·round_up(B·h·S·d·2, 256) bytes skips the
 *              last-wave balancing of attn_fwd_ws, and a size in between is
 *              rejected.  On return it holds the rounded copies of q, k, v,
 *              in that order, each at a 256-byte aligned offset.
 *   other arguments as attn_fwd; d in {64, 128}.
 *
 * Two launches on `stream`: one conversion kernel rounds q, k, v to
 * out_dtype (round to nearest even; fp16 overflows to inf above 65504), then
 * the fused kernel runs on the copies as attn_fwd_ws does.  Errors:
 * ATTN_E_NULL, ATTN_E_LAYOUT, ATTN_E_DTYPE (out_dtype), ATTN_E_SHAPE,
 * ATTN_E_ALIGN, ATTN_E_ALIAS, ATTN_E_WORKSPACE, ATTN_E_DEVICE, or a cudaError_t.
 */
int attn_fwd_mixed(const float* q, const float* k, const float* v, void* o, float* lse, int B, int h,
                   int S, int d, float scale, int layout, int out_dtype, void* workspace, size_t ws_bytes,
                   void* stream);

/* Workspace bytes attn_fwd_mixed needs on the current device (0 for invalid sizes). */
size_t attn_fwd_mixed_workspace_bytes(int B, int h, int S, int d, int out_dtype);

/*
 * attn_fwd_grouped -- attn_fwd on the third layout of "WebGPU 算子优化：QKV
 * 内存合并与 FlashAttention 分块计算", §QKV 矩阵的内存合并模式选择 ("split":
 * heads in groups, each group stored contiguously).  q, k, v, o are
 * [B, h/heads_per_group, S, heads_per_group, d]: per group, positions in
 * order and the group's heads interleaved within a position.
 * heads_per_group = 1 is the contiguous layout, = h the head-interleaved one.
 * 16-bit dtypes only (ATTN_E_DTYPE for ATTN_F32); heads_per_group must divide
 * h (ATTN_E_SHAPE).  Other arguments, lse and errors as attn_fwd.
 */
int attn_fwd_grouped(const void* q, const void* k, const void* v, void* o, float* lse, int B, int h,
                     int S, int d, int heads_per_group, float scale, int dtype, void* stream);

/*
 * attn_fwd_naive -- the unfused "standard" attention the pages compare
 * against: "Transformer算子生态深度分析" §2.5 materialises S and A in device
 * memory; the online-softmax proposal page ("[WebGPU] Proposal: Add an option
 * to use online softmax instead of naive softmax", §三) splits the softmax
 * into two dispatches.  Four launches:
 *   1. S = scale · Q·K^T  -> fp32 [B, h, S, S] in the workspace (tensor cores)
 *   2. pass 1: per row m = max S, l = sum exp(S - m)  (reads S)
 *   3. pass 2: P = exp(S - m) / l -> dtype [B, h, S, S] in the workspace (reads S)
 *   4. O = P·V (tensor cores)
 * Same arguments and result as attn_fwd, 16-bit dtypes only, plus a caller
 * workspace of at least attn_fwd_naive_workspace_bytes(B, h, S, dtype) bytes,
 * 256-byte aligned.  On return (after the stream completes) the workspace
 * holds S (fp32), then P (dtype), then the fp32 row statistics m and l.
 * Errors: as attn_fwd, plus ATTN_E_WORKSPACE.
 */
int attn_fwd_naive(const void* q, const void* k, const void* v, void* o, float* lse, int B, int h,
                   int S, int d, float scale, int layout, int dtype, void* workspace,
                   size_t ws_bytes, void* stream);
/* Workspace size for attn_fwd_naive: B·h·S²·(4 + elt) + 2·B·h·S·4 bytes, rounded
 * up to 256 B per part; 0 when the arguments are invalid. */
size_t attn_fwd_naive_workspace_bytes(int B, int h, int S, int dtype);

/*
 * qkv_proj_attn -- fused QKV projection followed by attention
 * ("Transformer算子生态深度分析" §2.1: one product with the concatenated weight
 * [D, 3D], then split into heads; then §2.2-§2.4).
 *
 *   x      [in]  [B, S, D] row-major, dtype ATTN_F16 or ATTN_BF16.
 *   w_qkv  [in]  [D, 3D] row-major; columns [0,D) produce Q, [D,2D) K,
 *                [2D,3D) V; within each third, column c belongs to head
 *                c / d, feature c % d (d = D / h).  No bias.
 *   o      [out] [B, S, h, d] (head-interleaved), same dtype.
 *   B, S, D, h   D must equal h·d with d in {64, 128}.
 *   workspace    at least qkv_proj_attn_workspace_bytes(B, S, D, dtype)
 *                bytes of device memory, 256-byte aligned.  On return it
 *                holds the projection [B, S, 3D] (dtype, rounded to
 *                nearest), i.e. Q, K, V in head-interleaved layout with row
 *                stride 3D, which the attention kernel reads in place.
 * Softmax scale is 1/sqrt(d).  Two launches (tensor-core GEMM, then the
 * attn_fwd kernel).  Errors: as attn_fwd, plus ATTN_E_WORKSPACE.
 */
int qkv_proj_attn(const void* x, const void* w_qkv, void* o, int B, int S, int D, int h, int dtype,
                  void* workspace, size_t ws_bytes, void* stream);
/* Workspace size for qkv_proj_attn: B·S·3D·elt bytes rounded up to 256; 0 when invalid. */
size_t qkv_proj_attn_workspace_bytes(int B, int S, int D, int dtype);

/*
 * qkv_proj_attn_fused -- the same result as qkv_proj_attn in ONE kernel
 * launch, with the projection feeding the attention on chip: the fusion of
 * "Transformer算子生态深度分析" §2.7 (算子层面的优化要点), the projected Q,
 * K, V going straight into the attention instead of through memory.  One
 * CTA per (batch, head) computes that head's K and V for all S positions
 * (fp32 in tensor memory, then rounded to the 16-bit type in shared memory),
 * then, 128 query rows at a time, Q and the online-softmax attention against
 * them.  Nothing but X, W_qkv and O touches device memory: no workspace.
 *
 *   x, w_qkv, o, B, S, D, h, dtype, stream   as for qkv_proj_attn.
 *
 * Supported sizes: d = D / h = 64 and 1 <= S <= 512 (one head's K and V must
 * fit in shared memory); other sizes return ATTN_E_SHAPE -- use
 * qkv_proj_attn.  The result equals qkv_proj_attn's up to fp32 summation
 * order (both round the projection to the 16-bit type before the attention).
 * Errors: as qkv_proj_attn without the workspace checks.
 */
int qkv_proj_attn_fused(const void* x, const void* w_qkv, void* o, int B, int S, int D, int h, int dtype,
                        void* stream);

/*
 * qkv_proj_attn_noalloc -- qkv_proj_attn for callers that cannot allocate
 * device memory.  The pages have no counterpart to this entry point.
 *
 * Some callers cannot call cudaMalloc (or any allocator) at the point where
 * they run attention: a plugin inside a host application that hands over only
 * its input and output buffers and owns every other byte of device memory; a
 * framework whose memory pool must account for all allocations; a
 * latency-critical loop that cannot afford an allocation's implicit device
 * synchronisation.  This entry point needs no workspace argument: the
 * [B, S, 3D] projection goes to a fixed scratch array of
 * ATTN_NOALLOC_SCRATCH_BYTES that the library declares statically in device
 * memory (every GPU that loads the library holds it until the process exits).
 * The call itself calls no allocator (see below for what the first call on a
 * device implies).
 *
 *   x, w_qkv, o, B, S, D, h, dtype, stream   as for qkv_proj_attn.
 *
 * Limit: B·S·3D·elt (rounded up to 256 bytes) must not exceed
 * ATTN_NOALLOC_SCRATCH_BYTES (32 MiB, e.g. B·S <= 7281 at D = 768 in fp16);
 * larger problems return ATTN_E_SCRATCH_LIMIT and launch nothing.
 * The first call on each device resolves the scratch array's device address
 * (with that device current).  Under CUDA's default lazy module loading, that
 * first call is also what loads the part of the library holding the array:
 * the driver then reserves its 32 MiB of device memory, which can fail with
 * cudaErrorMemoryAllocation (returned as a positive code) and may synchronise
 * the device.  So make the first call on each device during set-up, before any
 * stream capture and while memory is still free, or run the process with
 * CUDA_MODULE_LOADING=EAGER so that the array is reserved when the context is
 * created.  Every later call allocates nothing and does not synchronise.
 * All calls share the one array and it keeps the last call's
 * contents; nothing in it needs to start at zero because the projection
 * overwrites every element it later reads.  Calls that overlap on the GPU
 * (for example on two streams at once) race on the array: serialise them.
 * Errors: as qkv_proj_attn (without the workspace checks, and checked first),
 * plus ATTN_E_SCRATCH_LIMIT.
 */
#define ATTN_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)
int qkv_proj_attn_noalloc(const void* x, const void* w_qkv, void* o, int B, int S, int D, int h,
                          int dtype, void* stream);

/*
 * attn_select_kernel -- the softmax-strategy policy of the online-softmax
 * proposal page ("[WebGPU] Proposal: Add an option to use online softmax
 * instead of naive softmax", §六 select_kernel): the online (fused) kernel
 * when the option is enabled and seq_len exceeds the threshold, the naive
 * two-pass kernel otherwise.  threshold <= 0 selects the page's 1024.
 * Returns ATTN_KERNEL_ONLINE or ATTN_KERNEL_NAIVE.  Host only; no CUDA call.
 */
int attn_select_kernel(int option_enabled, int seq_len, int threshold);

/*
 * attn_fwd_auto -- attn_fwd or attn_fwd_naive, as attn_select_kernel picks
 * for (option_enabled, S, threshold).  Arguments as attn_fwd; `workspace` /
 * `ws_bytes` are needed only when the naive kernel is picked (size from
 * attn_fwd_naive_workspace_bytes; ATTN_E_WORKSPACE otherwise).  `chosen`
 * (may be NULL) receives the attn_kernel that ran.
 */
int attn_fwd_auto(const void* q, const void* k, const void* v, void* o, float* lse, int B, int h,
                  int S, int d, float scale, int layout, int dtype, int option_enabled,
                  int threshold, void* workspace, size_t ws_bytes, void* stream, int* chosen);

/*
 * attn_compare -- the numeric-agreement guard of the same page (§六
 * assert_numerically_equal): synchronises `stream`, then compares n elements
 * of two device buffers of `dtype` and writes max |a - b| to *max_abs
 * (host, may be NULL).  Returns ATTN_OK when it is <= atol, ATTN_E_MISMATCH
 * otherwise (a NaN counts as a mismatch), or an error.  The page uses
 * atol = 1e-3; for 16-bit outputs the two kernels also round P differently.
 * Each call accumulates into its own device result word (64 statically
 * declared words, taken in turn), so up to 64 calls may run at the same time
 * on different streams or host threads without sharing a result.
 */
int attn_compare(const void* a, const void* b, long long n, int dtype, float atol, float* max_abs,
                 void* stream);

/* Human-readable name of an ATTN_* status or a cudaError_t (positive). Never NULL. */
const char* attn_status_string(int status);

/*
 * attn_get_device_status -- synchronises `stream`, then returns and clears
 * the device status word of the current device: ATTN_OK, or ATTN_E_TIMEOUT
 * when a kernel gave up on a pipeline wait (its output is then undefined), or
 * a positive cudaError_t if the synchronisation itself failed.
 * `detail` (may be NULL) receives the raw code the kernel recorded
 * (kernel id << 24 | role << 16 | tile index), 0 if none.
 */
int attn_get_device_status(void* stream, unsigned int* detail);

/*
 * attn_selftest_wait_timeout -- diagnostics for the failure reporting above.
 * The pages have no counterpart; this exercises the library's own handling
 * of a stalled pipeline.  Launches one warp that waits on an mbarrier nothing
 * will ever arrive on, with the same bounded wait the attention kernels use
 * and a limit of `limit_cycles` SM clock cycles (1 .. 10^10).  The kernel
 * gives up after the limit, records detail code 15 << 24 | 1 << 16 in the
 * device status word and returns: attn_get_device_status then reports
 * ATTN_E_TIMEOUT, and the CUDA context stays usable.  No fault, trap or hang
 * is involved.  Errors: ATTN_E_SHAPE for a limit out of range, ATTN_E_DEVICE.
 */
int attn_selftest_wait_timeout(long long limit_cycles, void* stream);

/* ABI version of this header: 1. */
int attn_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_GB300_H */
