/*
 * vt_attn — scaled dot-product attention forward on one GB300 GPU (sm_103a).
 *
 * The operation (VeriTile page "VeriTile.Examples.FlashAttention1.NaiveRefinement":
 * fa1NaiveReference4D and fa1NaiveCausalReference4D, with the sequence-boundary and
 * head-dimension-tail write contract of fa1_boundaryD_refines_naive_reference_views;
 * separate query/key and value widths as in the accy page
 * "tiny.accy.kernel.library.attention", spec fields `qk` and `value`):
 *
 *   for every batch b < B, head h < H, query row i < S_q and value column e < D_v
 *     O[b,h,i,e] = sum_{j in A_i} softmax_j( scale * sum_{d<D_qk} Q[b,h,i,d] K[b,h,j,d] ) V[b,h,j,e]
 *   where A_i = { j < S_k } (causal = 0) or { j < S_k : j <= i } (causal != 0; key j
 *   <= query i counted from index 0 of both sequences).
 *
 * Layouts.  Q is [B,H,S_q,D_qk], K is [B,H,S_k,D_qk], V is [B,H,S_k,D_v] and O is
 * [B,H,S_q,D_v], the last index contiguous (stride 1).  vt_attn_fwd takes the packed
 * row-major layout; vt_attn_fwd_strided takes element strides for the (b, h, s)
 * indices of each tensor.  All four pointers are DEVICE pointers (CUDA global memory
 * of the current device).
 *
 * Element types.  VT_BF16: bf16 in, bf16 out, products accumulated in fp32 on the
 * tensor cores (probabilities are rounded to bf16 before the P*V product; the row sum
 * that normalises O counts each key tile's largest probability at its bf16 value, so a
 * row dominated by one key reproduces that key's value row up to the output rounding.
 * That holds for one dominating key per tile: when two or more keys of a tile carry most
 * of a row's weight, the bf16 rounding of the others' probabilities stays in the result,
 * an error of up to about 2^-9 of |O| on top of the output rounding; for |V| in [4, 8)
 * that is about 0.03).
 * VT_F32: fp32 in, fp32 out, products on the TF32 tensor-core path with fp32
 * accumulation (inputs and probabilities keep the TF32 subset of their bits).
 *
 * Ownership.  The caller owns every buffer.  The library allocates no device memory
 * per call: tensor maps are built on the host and passed by value to the kernel.
 *
 * Writes.  Only O's logical elements (i < S_q, e < D_v of each (b, h)) are written;
 * memory between rows or heads of a strided O is never touched.  O must not overlap
 * Q, K or V, and no two of O's logical elements may share an address (the strides may
 * nest the b, h and s indices in any order, e.g. [B,S,H,D], with any padding).
 *
 * Asynchrony.  Calls enqueue work on `stream` and return without waiting.  A kernel
 * that detects a problem on the device (a pipeline wait that exceeds its time limit)
 * records it in the device status word of the stream it was launched on instead of
 * faulting; vt_last_device_status(stream) synchronises that stream and returns (and
 * clears) that stream's status only.  If the environment variable VT_CHECK is set to a
 * non-zero value, every call does this itself.
 *
 * Argument errors are detected on the host before anything is launched:
 *   VT_ERR_INVALID_ARG   a NULL pointer, a negative extent, S_k, D_qk or D_v equal to 0,
 *                        an unknown dtype, a non-finite scale, O overlapping Q/K/V or
 *                        itself, a non-positive stride, or (vt_attn_fwd) extents whose
 *                        packed element count overflows 64 bits;
 *   VT_ERR_UNSUPPORTED   D_qk or D_v above 128, S_q or S_k above 2^30, B or H above
 *                        2^31 - 1, a (b, h, s) stride of 2^40 bytes or more (beyond a TMA
 *                        tensor map), or more than 2^31 - 1 work units (query blocks x heads x
 *                        batches x split-KV shares);
 *   (also VT_ERR_INVALID_ARG: extents and strides whose byte span overflows 64 bits);
 *   VT_ERR_MISALIGNED    a pointer not 16-byte aligned, or a (b, h, s) stride whose
 *                        byte size is not a multiple of 16 (the TMA engine's rule);
 *   VT_ERR_CUDA          a CUDA runtime or driver call failed (no device, launch error).
 * B, H or S_q equal to 0 is a valid empty problem: VT_OK, nothing launched.
 */
#ifndef VT_ATTN_H
#define VT_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st *vt_stream_t;

typedef enum { VT_F32 = 0, VT_BF16 = 1 } vt_dtype;

typedef enum {
    VT_OK = 0,
    VT_ERR_INVALID_ARG = 1,
    VT_ERR_UNSUPPORTED = 2,
    VT_ERR_MISALIGNED = 3,
    VT_ERR_CUDA = 4,
    VT_ERR_DEVICE_TIMEOUT = 5,
    VT_ERR_DEVICE_BOUNDS = 6
} vt_status;

/*
 * Attention forward on packed [B,H,S,D] tensors (the operation above).
 * Q, K, V: device pointers to the inputs (read only).  O: device pointer to the output.
 * scale: the factor applied to every dot product (the VeriTile reference's `scale`
 * parameter; 1/sqrt(D_qk) is the usual choice).  causal: 0 or non-zero.
 */
vt_status vt_attn_fwd(const void *Q, const void *K, const void *V, void *O,
                      int64_t B, int64_t H, int64_t S_q, int64_t S_k,
                      int64_t D_qk, int64_t D_v,
                      float scale, int causal, vt_dtype dtype, vt_stream_t stream);

/*
 * The same operation on strided tensors.  x_stride[0..2] are the element strides of
 * the b, h and s indices of tensor x; its last index has stride 1.  Every stride must
 * be positive and its byte size a multiple of 16.
 */
vt_status vt_attn_fwd_strided(const void *Q, const int64_t q_stride[3],
                              const void *K, const int64_t k_stride[3],
                              const void *V, const int64_t v_stride[3],
                              void *O, const int64_t o_stride[3],
                              int64_t B, int64_t H, int64_t S_q, int64_t S_k,
                              int64_t D_qk, int64_t D_v,
                              float scale, int causal, vt_dtype dtype, vt_stream_t stream);

/*
 * Options for vt_attn_fwd_ex.  A zeroed struct gives the defaults of vt_attn_fwd.
 *   wait_timeout_ns  limit for any single pipeline wait inside the kernel before it
 *                    gives up, records VT_ERR_DEVICE_TIMEOUT and exits cleanly
 *                    (0: 2 seconds).
 *   flags            VT_OPT_TEST_STALL makes the kernel wait on a barrier that is never
 *                    signalled, so that the time-limit path can be tested; it does no
 *                    attention work and leaves O unwritten.
 *                    VT_OPT_TEST_BOUNDS (debug library only, libvt_attn_debug.so, built
 *                    with VT_DEBUG) makes the first device index check of the producer
 *                    report a failure, so that the VT_ERR_DEVICE_BOUNDS path can be tested:
 *                    the kernel stops before any access and leaves O unwritten.  The
 *                    release library ignores it.
 *
 * The debug library exports the same entry points.  Its kernels check their index invariants
 * (decoded work units, key-tile ranges, ring slots, output rows) before each access they guard;
 * a failed check records VT_ERR_DEVICE_BOUNDS for vt_last_device_status, skips the access and
 * stops the kernel through the same clean path as a time-out.
 */
#define VT_OPT_TEST_STALL 1u
#define VT_OPT_TEST_BOUNDS 2u
typedef struct {
    uint64_t wait_timeout_ns;
    uint32_t flags;
    uint32_t reserved;
} vt_attn_opts;

/* vt_attn_fwd_strided with options (opts may be NULL). */
vt_status vt_attn_fwd_ex(const void *Q, const int64_t q_stride[3],
                         const void *K, const int64_t k_stride[3],
                         const void *V, const int64_t v_stride[3],
                         void *O, const int64_t o_stride[3],
                         int64_t B, int64_t H, int64_t S_q, int64_t S_k,
                         int64_t D_qk, int64_t D_v,
                         float scale, int causal, vt_dtype dtype,
                         const vt_attn_opts *opts, vt_stream_t stream);

/*
 * Split-KV forward: the same operation, with the key range of every query block cut into
 * n_split contiguous shares that separate CTAs process at the same time.  Each share writes an
 * unnormalised partial output with its row max, its row sum and that sum's correction for the
 * bf16 rounding of P (bf16 I/O) to `workspace`; a merge kernel then
 * combines the shares of each row into O (the continuation step of the VeriTile coverage table's
 * attention_fwd_triton3 row, case 4, which reads a previous M, L and Out and merges further keys).
 * It pays off when B * H * ceil(S_q / 256) is below the number of SMs (long keys, few queries).
 *
 *   n_split          1 .. 64; 1 is the plain forward (workspace unused, may be NULL).
 *   workspace        DEVICE memory owned by the caller, 256-byte aligned, at least
 *                    vt_attn_splitkv_workspace_size(B, H, S_q, D_v, n_split) bytes, not overlapping
 *                    Q, K, V or O.  Its contents are scratch: overwritten by every call, and two
 *                    calls that share a workspace must not overlap on the GPU.
 * Both element types (the fp32 shares cut 64-key tiles, the bf16 shares 128-key tiles).  Other
 * arguments and errors as for vt_attn_fwd_strided; a too small or NULL workspace is
 * VT_ERR_INVALID_ARG.
 */
vt_status vt_attn_fwd_splitkv(const void *Q, const int64_t q_stride[3],
                              const void *K, const int64_t k_stride[3],
                              const void *V, const int64_t v_stride[3],
                              void *O, const int64_t o_stride[3],
                              int64_t B, int64_t H, int64_t S_q, int64_t S_k,
                              int64_t D_qk, int64_t D_v,
                              float scale, int causal, vt_dtype dtype,
                              int n_split, void *workspace, size_t workspace_bytes,
                              vt_stream_t stream);

/* Bytes of workspace vt_attn_fwd_splitkv needs (0 when n_split <= 1, an extent is not positive, or
 * the size overflows: no such workspace can exist, and such a call is rejected).
 * Host-only arithmetic: no GPU call. */
size_t vt_attn_splitkv_workspace_size(int64_t B, int64_t H, int64_t S_q, int64_t D_v, int n_split);

/* The number of shares this library would pick on the current device: the most that still fit
 * one wave of CTAs with at least four key tiles each (128 keys for bf16, 64 for fp32); 1 when
 * splitting does not pay.  Queries the current device's SM count. */
int vt_attn_splitkv_choose(int64_t B, int64_t H, int64_t S_q, int64_t S_k, int causal, vt_dtype dtype);

/*
 * vt_attn_fwd_splitkv without a caller-provided workspace, for callers that cannot allocate
 * device memory: for example a plugin running inside a host framework that owns every byte of
 * device memory and does not let extensions call cudaMalloc, or a latency-critical service that
 * must not allocate after start-up because an allocation can block and synchronise the device.
 * The pages describe no such call; it has no counterpart in them.
 *
 * The shares' partial results live in a fixed 32 MiB array inside this library (a static
 * __device__ array: every GPU that loads the library holds it until the process exits).  The call
 * itself allocates nothing.  Arguments and errors are those of vt_attn_fwd_splitkv without the
 * workspace; in addition, a problem whose partial results need more than 32 MiB
 * (vt_attn_splitkv_workspace_size(B, H, S_q, D_v, n_split) > 33554432) is rejected with
 * VT_ERR_UNSUPPORTED before anything runs.  n_split = 1 uses no scratch at all.
 *
 * The first call with n_split > 1 on a device looks up the array's device address
 * (cudaGetSymbolAddress) and remembers it; make that first call before any stream capture.  All
 * calls share the one array, which keeps whatever the last call left there: every call writes all
 * the partial results it reads, so nothing has to start at zero, but calls that overlap on the GPU
 * (concurrent streams, or several host threads) race on the array and must be serialised by the
 * caller.
 */
vt_status vt_attn_fwd_splitkv_noalloc(const void *Q, const int64_t q_stride[3],
                                      const void *K, const int64_t k_stride[3],
                                      const void *V, const int64_t v_stride[3],
                                      void *O, const int64_t o_stride[3],
                                      int64_t B, int64_t H, int64_t S_q, int64_t S_k,
                                      int64_t D_qk, int64_t D_v,
                                      float scale, int causal, vt_dtype dtype,
                                      int n_split, vt_stream_t stream);

/*
 * General form.  Everything above is a special case of vt_attn_fwd_general, which adds:
 *
 * Grouped key/value heads (GQA; H_kv = 1 is multi-query attention).  K is [B,H_kv,S_k,D_qk] and V
 * is [B,H_kv,S_k,D_v]; query head h < H reads key/value head h / (H / H_kv), the num_kv_heads
 * indexing of the VeriTile coverage table's block-sparse attention row.  H must be a multiple of
 * H_kv; k_stride and v_stride are the strides of (b, h_kv, s).
 *
 * A mask choosing the keys A_i of query row i (o = offset >= 0, w = window >= 1):
 *   VT_MASK_NONE               A_i = { j < S_k }
 *   VT_MASK_CAUSAL             A_i = { j < S_k : j <= i + o }; query i sits at key position i + o
 *                              (the start_position of the coverage table's attention_llama causal
 *                              row; o = S_k - S_q aligns the last query with the last key)
 *   VT_MASK_WINDOW             A_i = { j < S_k : i + o - w < j <= i + o }: the w most recent keys
 *                              (the sliding window of the coverage table's attention_fwd_triton3
 *                              row, case 1)
 *   VT_MASK_WINDOW_COMPLEMENT  A_i = { j < S_k : j <= i + o - w }: the causal keys the window leaves
 *                              out (case 2 of the same row)
 * Key tiles outside every row's A_i are skipped, not masked.  A row whose A_i is empty (possible
 * with the window kinds only) is written as 0.
 *
 * An optional log-sum-exp output: lse, if not NULL, is a DEVICE fp32 array [B,H,S_q] (packed,
 * row-major) that receives LSE[b,h,i] = log(sum_{j in A_i} exp(scale * Q_i . K_j)), natural log,
 * -inf for an empty row.  With it, two calls over disjoint key sets (a window and its complement,
 * or two key ranges) combine into the call over their union: O = sum_k e^{LSE_k} O_k / sum_k e^{LSE_k}
 * (the continuation case 4 of the attention_fwd_triton3 row).  Must be 4-byte aligned and must not
 * overlap Q, K, V, O or the workspace.
 *
 * n_split, workspace and workspace_bytes are those of vt_attn_fwd_splitkv;
 * opts those of vt_attn_fwd_ex (may be NULL); mask may be NULL (VT_MASK_NONE).  Errors as for
 * vt_attn_fwd_splitkv, and VT_ERR_INVALID_ARG for H_kv < 1, H not a multiple of H_kv, an unknown mask
 * kind, offset < 0, window < 1 with a window kind, or a misplaced lse; VT_ERR_UNSUPPORTED for
 * offset or window above 2^40.
 */
typedef enum {
    VT_MASK_NONE = 0,
    VT_MASK_CAUSAL = 1,
    VT_MASK_WINDOW = 2,
    VT_MASK_WINDOW_COMPLEMENT = 3
} vt_mask_kind;

typedef struct {
    int32_t kind;     /* vt_mask_kind */
    int32_t reserved; /* 0 */
    int64_t offset;   /* o >= 0 */
    int64_t window;   /* w >= 1 for the window kinds; ignored otherwise */
} vt_attn_mask;

vt_status vt_attn_fwd_general(const void *Q, const int64_t q_stride[3],
                              const void *K, const int64_t k_stride[3],
                              const void *V, const int64_t v_stride[3],
                              void *O, const int64_t o_stride[3], float *lse,
                              int64_t B, int64_t H, int64_t H_kv, int64_t S_q, int64_t S_k,
                              int64_t D_qk, int64_t D_v, float scale, vt_dtype dtype,
                              const vt_attn_mask *mask, int n_split,
                              void *workspace, size_t workspace_bytes,
                              const vt_attn_opts *opts, vt_stream_t stream);

/* A static, human-readable name for a status code (never NULL). */
const char *vt_status_str(vt_status status);

/*
 * Synchronise `stream`, then return and clear the device status word that the kernels launched on
 * `stream` (on the current device) write: VT_OK, VT_ERR_DEVICE_TIMEOUT or VT_ERR_DEVICE_BOUNDS;
 * VT_ERR_CUDA if the synchronisation itself reports an error.  Other streams' words are neither read
 * nor cleared, and no other stream is waited for.
 *
 * Words are kept per stream handle: the first 255 distinct handles a process passes to this library get
 * a word each, in order of first use, and any later handle shares one common word (a destroyed stream's
 * handle keeps its word, which a new stream that receives the same handle inherits).  The per-thread
 * default stream is one handle for all threads.  A launch captured into a CUDA graph writes the word of
 * the stream it was captured on, whichever stream the graph is later launched into.
 */
vt_status vt_last_device_status(vt_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* VT_ATTN_H */
