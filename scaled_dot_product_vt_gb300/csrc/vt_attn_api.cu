// Host side of the vt_attn C ABI: argument checks, TMA tensor maps, launch.
//
// The operation and its argument contract are stated in include/vt_attn.h.  Nothing here
// touches the GPU before every argument has been checked.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <mutex>
#include <type_traits>

#include <nvtx3/nvToolsExt.h>

#include "../../include/vt_attn.h"
#include "vt_attn_bf16_2q.cuh"
#include "vt_attn_f32_2q.cuh"
#include "vt_attn_merge.cuh"

namespace vt {

// Device status words (kStatusTimeout, kStatusBounds), one per stream slot: a launch records what its
// kernels detect in the slot of the stream it was issued on, and vt_last_device_status reads only that
// stream's slot.  Slot 0 is shared by the streams beyond the table (kStatusSlots - 1 distinct streams).
constexpr int kStatusSlots = 256;
__device__ unsigned g_status[kStatusSlots];

// Scratch of vt_attn_fwd_splitkv_noalloc, for callers that cannot allocate device memory: a
// fixed array that exists on every GPU that loads this library, for as long as the process runs.
constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;  // 32 MiB
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

namespace {

// An NVTX range over one public call (named after the entry point), for profilers that record NVTX;
// without one attached, push and pop return at once.
struct NvtxRange {
    explicit NvtxRange(const char *name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange &) = delete;
    NvtxRange &operator=(const NvtxRange &) = delete;
};

constexpr int64_t kMaxD = 128;
constexpr int64_t kMaxExtent = 0x7FFFFFFF;  // B and H (their product is bounded by the work-unit count)
// S_q and S_k: the kernels form row and key indices a few tiles past an extent in 32-bit ints
constexpr int64_t kMaxSeq = int64_t(1) << 30;
constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;
constexpr int kSmemLimit = 232448;  // 227 KiB per CTA on sm_100-class parts

struct Span {
    uintptr_t lo, hi;  // [lo, hi) bytes touched by a tensor's logical elements
};

// The bytes a tensor's logical elements touch; false when the extent arithmetic overflows (no such
// tensor fits in an address space).  Extents and strides are positive here.
bool span_of(const void *p, const int64_t st[3], int64_t B, int64_t H, int64_t S, int64_t D, int elt, Span *out) {
    const int64_t n[3] = {B - 1, H - 1, S - 1};
    int64_t last = D - 1, t = 0, bytes = 0;
    for (int i = 0; i < 3; ++i)
        if (__builtin_mul_overflow(n[i], st[i], &t) || __builtin_add_overflow(last, t, &last)) return false;
    if (__builtin_add_overflow(last, int64_t(1), &bytes) || __builtin_mul_overflow(bytes, int64_t(elt), &bytes))
        return false;
    const uintptr_t lo = reinterpret_cast<uintptr_t>(p);
    if (static_cast<uint64_t>(bytes) > UINTPTR_MAX - lo) return false;
    *out = {lo, lo + static_cast<uintptr_t>(bytes)};
    return true;
}

// The LSE array: B * H * S_q floats from `lse`; false on overflow.
bool lse_span(const float *lse, int64_t B, int64_t H, int64_t S_q, Span *out) {
    int64_t n = 0;
    if (__builtin_mul_overflow(B, H, &n) || __builtin_mul_overflow(n, S_q, &n) ||
        __builtin_mul_overflow(n, int64_t(sizeof(float)), &n))
        return false;
    const uintptr_t lo = reinterpret_cast<uintptr_t>(lse);
    if (static_cast<uint64_t>(n) > UINTPTR_MAX - lo) return false;
    *out = {lo, lo + static_cast<uintptr_t>(n)};
    return true;
}

// Largest (b, h, s) stride in bytes that a TMA tensor map accepts is below 2^40.
constexpr int64_t kMaxStrideBytes = int64_t(1) << 40;

bool overlap(Span a, Span b) { return a.lo < b.hi && b.lo < a.hi; }

bool env_check() {
    static const bool on = [] {
        const char *v = std::getenv("VT_CHECK");
        return v && v[0] && !(v[0] == '0' && v[1] == 0);
    }();
    return on;
}

// Per-device facts that do not change while the process runs, looked up once: the SM count, the L2
// size and the device address of the status words.
struct DeviceInfo {
    bool ready = false;
    int sms = 0;
    long long l2_bytes = 0;
    unsigned *status = nullptr;  // g_status on this device
};
constexpr int kMaxDevices = 64;
std::mutex g_info_mu;
DeviceInfo g_info[kMaxDevices];
struct SmemGrant {
    const void *kern;
    int dev;
    int bytes;
};
SmemGrant g_grants[64];
int g_n_grants = 0;

bool device_info(int dev, DeviceInfo *out) {
    if (dev < 0 || dev >= kMaxDevices) return false;
    std::lock_guard<std::mutex> lock(g_info_mu);
    DeviceInfo &d = g_info[dev];
    if (!d.ready) {
        void *status_ptr = nullptr;
        if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return false;
        int l2 = 0;
        if (cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev) != cudaSuccess) return false;
        d.l2_bytes = l2;
        if (cudaGetSymbolAddress(&status_ptr, g_status) != cudaSuccess) return false;
        d.status = static_cast<unsigned *>(status_ptr);
        d.ready = true;
    }
    *out = d;
    return true;
}

// The status slot of a stream: the first kStatusSlots - 1 distinct stream handles seen get slots 1, 2, ...
// in order of first use; later ones share slot 0.  Handles are process-wide, so one table serves every
// device (each device has its own array of words).
std::mutex g_slot_mu;
cudaStream_t g_slot_stream[kStatusSlots];
int g_n_slots = 1;

int status_slot(cudaStream_t s) {
    std::lock_guard<std::mutex> lock(g_slot_mu);
    for (int i = 1; i < g_n_slots; ++i)
        if (g_slot_stream[i] == s) return i;
    if (g_n_slots == kStatusSlots) return 0;
    g_slot_stream[g_n_slots] = s;
    return g_n_slots++;
}

// cudaFuncSetAttribute for the dynamic shared memory size, only when a kernel needs more on a
// device than it was granted before.
bool ensure_smem(const void *kern, int dev, int bytes) {
    std::lock_guard<std::mutex> lock(g_info_mu);
    for (int i = 0; i < g_n_grants; ++i)
        if (g_grants[i].kern == kern && g_grants[i].dev == dev) {
            if (g_grants[i].bytes >= bytes) return true;
            if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess)
                return false;
            g_grants[i].bytes = bytes;
            return true;
        }
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess) return false;
    if (g_n_grants < 64) g_grants[g_n_grants++] = {kern, dev, bytes};
    return true;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

// 4-D map over [B][H][S][D] (D innermost), box = 128-byte chunk of D x `rows` rows of S.
bool make_map(CUtensorMap *map, const void *ptr, const int64_t st[3], int64_t B, int64_t H, int64_t S, int64_t D,
              int elt, int rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(S), static_cast<cuuint64_t>(H),
                                static_cast<cuuint64_t>(B)};
    const cuuint64_t strides[3] = {static_cast<cuuint64_t>(st[2] * elt), static_cast<cuuint64_t>(st[1] * elt),
                                   static_cast<cuuint64_t>(st[0] * elt)};
    const cuuint32_t box[4] = {static_cast<cuuint32_t>(128 / elt), static_cast<cuuint32_t>(rows), 1, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    const CUresult r = fn(map, elt == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4,
                          const_cast<void *>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Workspace of a split-KV call: partial outputs, then row maxima, row sums and row-sum corrections
// (each part 256-byte aligned).
struct SplitLayout {
    size_t o_off, m_off, l_off, c_off, bytes;
};
// bytes = 0 when the sizes overflow (no such workspace can exist).
SplitLayout split_layout(int64_t B, int64_t H, int64_t S_q, int64_t D_v, int n_split) {
    auto up = [](uint64_t x) { return (x + 255) & ~uint64_t(255); };
    SplitLayout L{};
    uint64_t rows = 0, per = 0, o_bytes = 0;
    if (B <= 0 || H <= 0 || S_q <= 0 || D_v <= 0 || n_split <= 0 ||
        __builtin_mul_overflow(uint64_t(B), uint64_t(H), &rows) || __builtin_mul_overflow(rows, uint64_t(S_q), &rows) ||
        __builtin_mul_overflow(rows, uint64_t(n_split) * sizeof(float), &per) ||
        __builtin_mul_overflow(per, uint64_t(D_v), &o_bytes) || o_bytes > (uint64_t(1) << 60) ||
        per > (uint64_t(1) << 60))
        return L;
    L.o_off = 0;
    L.m_off = up(o_bytes);
    L.l_off = L.m_off + up(per);
    L.c_off = L.l_off + up(per);
    L.bytes = L.c_off + up(per);
    return L;
}

// One forward problem as the general entry point states it (include/vt_attn.h).
struct Problem {
    const void *Q, *K, *V;
    void *O;
    const int64_t *qs, *ks, *vs, *os;  // (b, h, s) element strides; K and V count key/value heads
    float *lse;                        // nullptr or [B*H*S_q]
    int64_t B, H, H_kv, S_q, S_k, D_qk, D_v;
    float scale;
    vt_dtype dtype;
    int mask;
    int64_t offset, window;
};

constexpr int64_t kMaxBandArg = int64_t(1) << 40;

// The band [i + lo, i + hi] of each mask kind, and whether later query blocks carry more work.
void band_of(const Problem &P, long long *lo, long long *hi, int *reverse) {
    switch (P.mask) {
        case VT_MASK_CAUSAL: *lo = -kBandInf; *hi = P.offset; *reverse = 1; return;
        case VT_MASK_WINDOW: *lo = P.offset - P.window + 1; *hi = P.offset; *reverse = 0; return;
        case VT_MASK_WINDOW_COMPLEMENT: *lo = -kBandInf; *hi = P.offset - P.window; *reverse = 1; return;
        default: *lo = -kBandInf; *hi = kBandInf; *reverse = 0; return;
    }
}

// Combine the n_split partial results of every row into O (and the LSE if asked for).
template <int ELT>
vt_status merge(const AttnParams &p, const Problem &P, cudaStream_t stream) {
    MergeParams mp{};
    mp.part_o = p.part_o;
    mp.part_m = p.part_m;
    mp.part_l = p.part_l;
    mp.part_c = p.part_c;
    mp.O = P.O;
    mp.lse = P.lse;
    mp.rows = P.B * P.H * P.S_q;
    mp.H = static_cast<int>(P.H);
    mp.S_q = static_cast<int>(P.S_q);
    mp.D_v = static_cast<int>(P.D_v);
    mp.n_split = p.n_split;
    mp.o_sb = P.os[0];
    mp.o_sh = P.os[1];
    mp.o_ss = P.os[2];
    const long long blocks = (mp.rows + kMergeRowsPerBlock - 1) / kMergeRowsPerBlock;
    if (blocks > 0x7FFFFFFFll) return VT_ERR_UNSUPPORTED;
    attn_merge_kernel<ELT><<<static_cast<unsigned>(blocks), 32 * kMergeRowsPerBlock, 0, stream>>>(mp);
    return cudaGetLastError() == cudaSuccess ? VT_OK : VT_ERR_CUDA;
}

// Per element type: bytes per element, keys per K/V tile and the MMA K-step (bf16 16, tf32 8).
template <int DT>
struct Elt {
    static constexpr int kElt = DT == kBF16 ? 2 : 4;
    static constexpr int kBN = DT == kBF16 ? q2::kBN : f2::kBN;
    static constexpr int kKStep = DT == kBF16 ? 16 : 8;
    static constexpr int kChunkElems = 128 / kElt;  // elements per 128-byte chunk
};

// A cluster size for the fp32 kernel: the most CTAs (8, 4 or 2) that may share one unit's key tiles while
// every CTA of the launch still fits one wave and keeps two key tiles or more; 1 when that does not pay.
int f32_cluster_size(long long units, long long key_tiles, int sms) {
    for (int c = f2::kMaxCluster; c >= 2; c /= 2)
        if (units * c <= sms && key_tiles >= 2LL * c) return c;
    return 1;
}

template <int DT>
vt_status launch(const Problem &P, const vt_attn_opts *opts, int n_split, void *workspace, cudaStream_t stream) {
    using C = Elt<DT>;
    const void *Q = P.Q, *K = P.K, *V = P.V;
    void *O = P.O;
    const int64_t *qs = P.qs, *ks = P.ks, *vs = P.vs, *os = P.os;
    const int64_t B = P.B, H = P.H, S_q = P.S_q, S_k = P.S_k, D_qk = P.D_qk, D_v = P.D_v;
    CUtensorMap tq, tk, tv;
    // K/V boxes are one key tile high
    const int kv_rows = DT == kBF16 ? q2::kBN : C::kBN;
    if (!make_map(&tq, Q, qs, B, H, S_q, D_qk, C::kElt, kBM) ||
        !make_map(&tk, K, ks, B, P.H_kv, S_k, D_qk, C::kElt, kv_rows))
        return VT_ERR_CUDA;
    // (fp32: Q is read by the kernel's softmax threads, which write it into TMEM)
    if (!make_map(&tv, V, vs, B, P.H_kv, S_k, D_v, C::kElt, kv_rows)) return VT_ERR_CUDA;

    AttnParams p{};
    p.B = static_cast<int>(B);
    p.H = static_cast<int>(H);
    p.S_q = static_cast<int>(S_q);
    p.S_k = static_cast<int>(S_k);
    p.D_qk = static_cast<int>(D_qk);
    p.D_v = static_cast<int>(D_v);
    p.n_qblocks = static_cast<int>((S_q + kBM - 1) / kBM);
    p.qk_ksteps = static_cast<int>((D_qk + C::kKStep - 1) / C::kKStep);
    p.q_chunks = static_cast<int>((D_qk + C::kChunkElems - 1) / C::kChunkElems);
    p.v_chunks = static_cast<int>((D_v + C::kChunkElems - 1) / C::kChunkElems);
    p.n_pv = static_cast<int>((D_v + 15) / 16 * 16);
    band_of(P, &p.band_lo, &p.band_hi, &p.reverse_q);
    p.kv_group = static_cast<int>(H / P.H_kv);
    p.lse = P.lse;
    p.scale_log2 = P.scale * 1.4426950408889634f;
    p.O = O;
    p.o_sb = os[0];
    p.o_sh = os[1];
    p.o_ss = os[2];
    p.o_vec32 = (reinterpret_cast<uintptr_t>(O) % 32 == 0 && (os[0] * C::kElt) % 32 == 0 &&
                 (os[1] * C::kElt) % 32 == 0 && (os[2] * C::kElt) % 32 == 0)
                    ? 1
                    : 0;
    p.V = V;
    p.v_sb = vs[0];
    p.v_sh = vs[1];
    p.v_ss = vs[2];
    p.Q = Q;
    p.q_sb = qs[0];
    p.q_sh = qs[1];
    p.q_ss = qs[2];
    p.tiles_per_unit = 2;
    p.cluster = 1;
    p.n_split = n_split;
    if (n_split > 1) {
        const SplitLayout L = split_layout(B, H, S_q, D_v, n_split);
        uint8_t *ws = static_cast<uint8_t *>(workspace);
        p.part_o = reinterpret_cast<float *>(ws + L.o_off);
        p.part_m = reinterpret_cast<float *>(ws + L.m_off);
        p.part_l = reinterpret_cast<float *>(ws + L.l_off);
        p.part_c = reinterpret_cast<float *>(ws + L.c_off);
    }
    p.timeout_ns = (opts && opts->wait_timeout_ns) ? opts->wait_timeout_ns : kDefaultTimeoutNs;
    p.flags = opts ? opts->flags : 0u;

    int dev = 0;
    DeviceInfo info;
    if (cudaGetDevice(&dev) != cudaSuccess || !device_info(dev, &info)) return VT_ERR_CUDA;
    p.status = info.status + status_slot(stream);
    const int sms = info.sms;

    if constexpr (DT == kBF16) {
        // two 128-row query tiles per CTA, 128-key tiles through a ring of equal K/V slots
        p.n_qblocks = static_cast<int>((S_q + q2::kRows - 1) / q2::kRows);
        const int q_bytes = 2 * p.q_chunks * static_cast<int>(q2::kChunkBytes);
        const int slot_bytes = (p.q_chunks > p.v_chunks ? p.q_chunks : p.v_chunks) * static_cast<int>(q2::kChunkBytes);
        const int budget = kSmemLimit - 1024 - static_cast<int>(sizeof(q2::Ctl)) - 256;
        p.stages = (budget - q_bytes) / slot_bytes;  // number of slots
        if (p.stages > q2::kMaxSlots) p.stages = q2::kMaxSlots;
        if (p.stages < 2) return VT_ERR_UNSUPPORTED;
        const int smem = 1024 + q_bytes + p.stages * slot_bytes;
        // Interleave the query blocks of about two waves' worth of heads, so the CTAs in flight
        // share their heads' K and V in L2, but no more heads than three quarters of L2 holds K and
        // V for: otherwise a head's blocks fall into different waves and its K/V is read again.
        const long long bh = B * H;
        long long grp = (2LL * sms + p.n_qblocks - 1) / p.n_qblocks;
        // (consecutive query heads share one K/V head when H_kv < H)
        const long long kv_head_bytes = S_k * (D_qk + D_v) * C::kElt;
        const long long l2_heads =
            info.l2_bytes > 0 ? (3 * info.l2_bytes / 4) / kv_head_bytes * (H / P.H_kv) : grp;
        if (grp > l2_heads) grp = l2_heads;
        p.head_group = static_cast<int>(grp < 1 ? 1 : (grp > bh ? bh : grp));
        const long long units = static_cast<long long>(p.n_qblocks) * bh * n_split;
        if (units > 0x7FFFFFFFll) return VT_ERR_UNSUPPORTED;
        p.n_units = static_cast<int>(units);
        // one CTA per unit; the shared memory admits one per SM, and a running CTA takes over the units of
        // the CTAs that have not started (cluster launch control), so about one per SM runs
        const unsigned grid = static_cast<unsigned>(units);
        // Q K^T K-steps of 16, rounded up to an even count (the TMA zero-fills past D_qk)
        const int ksteps = static_cast<int>((D_qk + 15) / 16);
        // value widths up to 64 leave TMEM room for the score ring (S of the next key tile during the softmax)
        const bool ring = p.n_pv <= 64;
        // kernel variants: K-steps of Q K^T, the score ring, the epilogue (O in any layout with the log-sum-exp;
        // partial outputs for a split-KV merge; O alone in 32-byte rows of whole 16-column groups), and a positive
        // scale folded into the exponent
        using Kern = void (*)(const CUtensorMap, const CUtensorMap, const CUtensorMap, const AttnParams);
        auto pick = [&](auto ring_c, auto epi_c, auto fold_c) -> Kern {
            constexpr bool R = decltype(ring_c)::value, F = decltype(fold_c)::value;
            constexpr int E = decltype(epi_c)::value;
            return ksteps <= 2   ? attn_fwd_bf16_2q_kernel<2, R, E, F>
                   : ksteps <= 4 ? attn_fwd_bf16_2q_kernel<4, R, E, F>
                   : ksteps <= 6 ? attn_fwd_bf16_2q_kernel<6, R, E, F>
                                 : attn_fwd_bf16_2q_kernel<8, R, E, F>;
        };
        using T_ = std::true_type;
        using F_ = std::false_type;
        using Plain = std::integral_constant<int, q2::kEpiPlain>;
        using Split = std::integral_constant<int, q2::kEpiSplit>;
        using Fast = std::integral_constant<int, q2::kEpiPlainFast>;
        const bool fold = p.scale_log2 > 0.0f;
        // (the short epilogue measured faster in the two-tile kernel and slower with the score ring)
        const int epi = n_split > 1 ? q2::kEpiSplit
                        : (fold && !ring && p.o_vec32 && D_v % 16 == 0 && !P.lse) ? q2::kEpiPlainFast
                                                                                : q2::kEpiPlain;
        Kern kern;
        if (fold) {
            kern = epi == q2::kEpiSplit       ? (ring ? pick(T_{}, Split{}, T_{}) : pick(F_{}, Split{}, T_{}))
                   : epi == q2::kEpiPlainFast ? pick(F_{}, Fast{}, T_{})
                                              : (ring ? pick(T_{}, Plain{}, T_{}) : pick(F_{}, Plain{}, T_{}));
        } else {
            kern = epi == q2::kEpiSplit ? (ring ? pick(T_{}, Split{}, F_{}) : pick(F_{}, Split{}, F_{}))
                                        : (ring ? pick(T_{}, Plain{}, F_{}) : pick(F_{}, Plain{}, F_{}));
        }
        if (!ensure_smem(reinterpret_cast<const void *>(kern), dev, smem)) return VT_ERR_CUDA;
        kern<<<grid, q2::kThreads, smem, stream>>>(tq, tk, tv, p);
        if (cudaGetLastError() != cudaSuccess) return VT_ERR_CUDA;
        if (n_split > 1) return merge<2>(p, P, stream);
        return VT_OK;
    } else {
        // fp32 I/O on the TF32 path: units of two 128-row query tiles when TMEM holds both tiles' S, O and Q
        // (D_qk rounded up to 8 plus D_v rounded up to 16 at most 192), else one; one CTA per unit and share.
        const int dq = p.qk_ksteps * 8;
        const int stage_bytes = (p.q_chunks + p.v_chunks) * f2::kBN * 128 + p.n_pv * f2::kBN * 4;
        const int budget = kSmemLimit - 1024 - static_cast<int>(sizeof(f2::Ctl)) - 256;
        p.stages = budget / stage_bytes;
        if (p.stages > f2::kMaxStages) p.stages = f2::kMaxStages;
        // The Q tiles arrive in the last stages' memory, and at least one stage must stay outside it: two tiles
        // when that fits and TMEM holds both tiles' S, O and Q, else one.
        auto q_stages = [&](int tiles) { return (tiles * p.q_chunks * kBM * 128 + stage_bytes - 1) / stage_bytes; };
        int T = 2 * (f2::kBN + p.n_pv + dq) <= 512 && p.stages >= q_stages(2) + 1 ? 2 : 1;
        if (p.stages < 2 || p.stages < q_stages(T) + 1) return VT_ERR_UNSUPPORTED;
        p.tiles_per_unit = T;
        p.n_qblocks = static_cast<int>((S_q + kBM * T - 1) / (kBM * T));
        const long long units = static_cast<long long>(p.n_qblocks) * B * H;
        // Without a caller's split, a unit's key tiles may be shared by the CTAs of a cluster, which merge
        // their results in distributed shared memory; the partials each CTA receives reuse its K/V ring.
        int cl = 1;
        if (n_split == 1) {
            const long long key_tiles = (S_k + f2::kBN - 1) / f2::kBN;
            cl = f32_cluster_size(units, key_tiles, sms);
            while (cl > 4 * T) cl /= 2;  // each CTA owns whole warps of rows (T * 128 / cl >= 32) in the merge
            // the merge stages every row of the unit and receives the other CTAs' rows in the ring's memory
            const long long merge_bytes = 2LL * T * kBM * ((D_v + 3) / 4 + 1) * 16;
            if (merge_bytes > static_cast<long long>(p.stages) * stage_bytes) cl = 1;
        }
        p.cluster = cl;
        // Without a cluster or shares the ring needs no more stages than the key tiles plus the Q tiles take
        // (a problem of a few key tiles then asks for far less shared memory).
        if (cl == 1 && n_split == 1) {
            const long long need = (S_k + f2::kBN - 1) / f2::kBN + q_stages(T);
            if (need < p.stages) p.stages = static_cast<int>(need < 2 ? 2 : need);
        }
        const long long ctas = units * (cl > 1 ? cl : n_split);
        if (ctas > 0x7FFFFFFFll) return VT_ERR_UNSUPPORTED;
        p.n_units = static_cast<int>(units);
        const int smem = 1024 + p.stages * stage_bytes;
        // Q K^T K-steps, and a positive scale folded into the exponent (a variant without the scores' scaling)
        using Kern = void (*)(const CUtensorMap, const CUtensorMap, const CUtensorMap, const AttnParams);
        auto pick = [&](auto fold_c) -> Kern {
            constexpr bool F = decltype(fold_c)::value;
            return dq <= 32   ? attn_fwd_f32_2q_kernel<4, F>
                   : dq <= 64 ? attn_fwd_f32_2q_kernel<8, F>
                   : dq <= 96 ? attn_fwd_f32_2q_kernel<12, F>
                              : attn_fwd_f32_2q_kernel<16, F>;
        };
        const Kern kern = p.scale_log2 > 0.0f ? pick(std::true_type{}) : pick(std::false_type{});
        if (!ensure_smem(reinterpret_cast<const void *>(kern), dev, smem)) return VT_ERR_CUDA;
        cudaLaunchConfig_t cfg{};
        cfg.gridDim = dim3(static_cast<unsigned>(ctas), 1, 1);
        cfg.blockDim = dim3(f2::kThreads, 1, 1);
        cfg.dynamicSmemBytes = static_cast<size_t>(smem);
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = static_cast<unsigned>(cl);
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = cl > 1 ? 1 : 0;
        if (cudaLaunchKernelEx(&cfg, kern, tq, tk, tv, p) != cudaSuccess) return VT_ERR_CUDA;
        if (cudaGetLastError() != cudaSuccess) return VT_ERR_CUDA;
        if (n_split > 1) return merge<4>(p, P, stream);
        return VT_OK;
    }
}

// Device address of g_noalloc_scratch on the current device (nullptr on failure).  The host-side
// name of the array is only a stand-in, so the address is looked up with cudaGetSymbolAddress,
// once per device with that device current, and remembered.
void *noalloc_scratch(int dev) {
    static void *addr[kMaxDevices] = {};
    if (dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_info_mu);
    if (!addr[dev]) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess) return nullptr;
        addr[dev] = ptr;
    }
    return addr[dev];
}

// Wait for `stream`, then read and clear the status word of its slot on the current device.  The read and
// the clear are ordered on `stream` itself, so no other stream is waited for.
vt_status read_status(cudaStream_t stream) {
    int dev = 0;
    DeviceInfo info;
    if (cudaGetDevice(&dev) != cudaSuccess || !device_info(dev, &info)) return VT_ERR_CUDA;
    unsigned *word = info.status + status_slot(stream);
    unsigned w = 0;
    if (cudaMemcpyAsync(&w, word, sizeof w, cudaMemcpyDeviceToHost, stream) != cudaSuccess) return VT_ERR_CUDA;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return VT_ERR_CUDA;
    if (w && cudaMemsetAsync(word, 0, sizeof w, stream) != cudaSuccess) return VT_ERR_CUDA;
    if (w & kStatusTimeout) return VT_ERR_DEVICE_TIMEOUT;
    if (w & kStatusBounds) return VT_ERR_DEVICE_BOUNDS;
    return VT_OK;
}

}  // namespace
}  // namespace vt

extern "C" {

const char *vt_status_str(vt_status s) {
    switch (s) {
        case VT_OK: return "VT_OK";
        case VT_ERR_INVALID_ARG: return "VT_ERR_INVALID_ARG: invalid argument";
        case VT_ERR_UNSUPPORTED: return "VT_ERR_UNSUPPORTED: shape not supported (D_qk, D_v <= 128; extents < 2^31)";
        case VT_ERR_MISALIGNED: return "VT_ERR_MISALIGNED: pointers must be 16-byte aligned and strides 16-byte multiples";
        case VT_ERR_CUDA: return "VT_ERR_CUDA: a CUDA runtime or driver call failed";
        case VT_ERR_DEVICE_TIMEOUT: return "VT_ERR_DEVICE_TIMEOUT: a kernel pipeline wait exceeded its time limit";
        case VT_ERR_DEVICE_BOUNDS: return "VT_ERR_DEVICE_BOUNDS: a kernel index check failed";
    }
    return "unknown vt_status";
}

vt_status vt_last_device_status(vt_stream_t stream) {
    const vt::NvtxRange range("vt_last_device_status");
    return vt::read_status(reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"

namespace vt {
namespace {

// The checks of include/vt_attn.h that need only the extents and scalars (in the header's order of
// precedence); VT_OK with *empty = true for a valid empty problem.
vt_status check_shape(const Problem &P, bool *empty) {
    *empty = false;
    const int64_t B = P.B, H = P.H, H_kv = P.H_kv, S_q = P.S_q, S_k = P.S_k, D_qk = P.D_qk, D_v = P.D_v;
    if (P.dtype != VT_F32 && P.dtype != VT_BF16) return VT_ERR_INVALID_ARG;
    if (B < 0 || H < 0 || S_q < 0 || S_k < 0 || D_qk < 0 || D_v < 0) return VT_ERR_INVALID_ARG;
    if (S_k == 0 || D_qk == 0 || D_v == 0) return VT_ERR_INVALID_ARG;
    if (H_kv < 1 || (H > 0 && H % H_kv != 0)) return VT_ERR_INVALID_ARG;
    if (!std::isfinite(P.scale)) return VT_ERR_INVALID_ARG;
    if (P.mask < VT_MASK_NONE || P.mask > VT_MASK_WINDOW_COMPLEMENT || P.offset < 0) return VT_ERR_INVALID_ARG;
    const bool windowed = P.mask == VT_MASK_WINDOW || P.mask == VT_MASK_WINDOW_COMPLEMENT;
    if (windowed && P.window < 1) return VT_ERR_INVALID_ARG;
    if (P.offset > vt::kMaxBandArg || (windowed && P.window > vt::kMaxBandArg)) return VT_ERR_UNSUPPORTED;
    if (D_qk > vt::kMaxD || D_v > vt::kMaxD) return VT_ERR_UNSUPPORTED;
    if (B > vt::kMaxExtent || H > vt::kMaxExtent || S_q > vt::kMaxSeq || S_k > vt::kMaxSeq)
        return VT_ERR_UNSUPPORTED;
    if (B == 0 || H == 0 || S_q == 0) *empty = true;
    return VT_OK;
}

// True when no two logical elements of a [B, H, S, D] tensor with (b, h, s) strides st and unit stride
// along D share an address: with the extents of size 1 left out and the rest taken in order of
// increasing stride, each stride reaches past everything the smaller ones span.  This accepts every
// nesting of the three indices ([B,H,S,D], [B,S,H,D], ...) without gaps or overlap, and any padding.
bool rows_disjoint(const int64_t st[3], int64_t B, int64_t H, int64_t S, int64_t D) {
    int64_t n[3] = {B, H, S}, s[3] = {st[0], st[1], st[2]};
    for (int i = 0; i < 3; ++i)  // insertion sort by stride
        for (int j = i; j > 0 && s[j] < s[j - 1]; --j) {
            const int64_t ts = s[j], tn = n[j];
            s[j] = s[j - 1]; n[j] = n[j - 1];
            s[j - 1] = ts; n[j - 1] = tn;
        }
    int64_t span = D;  // elements covered by the dimensions taken so far, as one contiguous extent
    for (int i = 0; i < 3; ++i) {
        if (n[i] <= 1) continue;
        if (s[i] < span) return false;
        int64_t t = 0;
        if (__builtin_mul_overflow(n[i] - 1, s[i], &t) || __builtin_add_overflow(span, t, &span)) return false;
    }
    return true;
}

// The checks of include/vt_attn.h on pointers, strides and the memory they describe (after check_shape
// passed on a non-empty problem).
vt_status check_memory(const Problem &P) {
    const int64_t B = P.B, H = P.H, H_kv = P.H_kv, S_q = P.S_q, S_k = P.S_k, D_qk = P.D_qk, D_v = P.D_v;
    if (!P.Q || !P.K || !P.V || !P.O || !P.qs || !P.ks || !P.vs || !P.os) return VT_ERR_INVALID_ARG;
    const int elt = P.dtype == VT_BF16 ? 2 : 4;
    const int64_t *st[4] = {P.qs, P.ks, P.vs, P.os};
    for (const int64_t *s : st)
        for (int i = 0; i < 3; ++i)
            if (s[i] <= 0) return VT_ERR_INVALID_ARG;
    const void *ptrs[4] = {P.Q, P.K, P.V, P.O};
    for (const void *ptr : ptrs)
        if (reinterpret_cast<uintptr_t>(ptr) % 16) return VT_ERR_MISALIGNED;
    for (const int64_t *s : st)
        for (int i = 0; i < 3; ++i)
            if (s[i] >= vt::kMaxStrideBytes / elt) return VT_ERR_UNSUPPORTED;
    for (const int64_t *s : st)
        for (int i = 0; i < 3; ++i)
            if ((s[i] * elt) % 16) return VT_ERR_MISALIGNED;
    vt::Span sq, sk, sv, so;
    if (!vt::span_of(P.Q, P.qs, B, H, S_q, D_qk, elt, &sq) || !vt::span_of(P.K, P.ks, B, H_kv, S_k, D_qk, elt, &sk) ||
        !vt::span_of(P.V, P.vs, B, H_kv, S_k, D_v, elt, &sv) || !vt::span_of(P.O, P.os, B, H, S_q, D_v, elt, &so))
        return VT_ERR_INVALID_ARG;
    if (vt::overlap(so, sq) || vt::overlap(so, sk) || vt::overlap(so, sv)) return VT_ERR_INVALID_ARG;
    // every output element has an address of its own (several CTAs would otherwise race on one)
    if (!vt::rows_disjoint(P.os, B, H, S_q, D_v)) return VT_ERR_INVALID_ARG;
    if (P.lse) {
        if (reinterpret_cast<uintptr_t>(P.lse) % 4) return VT_ERR_INVALID_ARG;
        vt::Span sl;
        if (!vt::lse_span(P.lse, B, H, S_q, &sl)) return VT_ERR_INVALID_ARG;
        if (vt::overlap(sl, sq) || vt::overlap(sl, sk) || vt::overlap(sl, sv) || vt::overlap(sl, so))
            return VT_ERR_INVALID_ARG;
    }
    return VT_OK;
}

// Every argument check shared by the forward entry points; VT_OK with *empty = true for a valid empty
// problem.
vt_status check_args(const Problem &P, bool *empty) {
    const vt_status r = check_shape(P, empty);
    if (r != VT_OK || *empty) return r;
    return check_memory(P);
}

// Checks of a split-KV workspace (n_split > 1): present, large enough, 256-byte aligned and clear of
// every tensor of the call.
vt_status check_workspace(const Problem &P, int n_split, const void *workspace, size_t workspace_bytes) {
    const size_t need = vt::split_layout(P.B, P.H, P.S_q, P.D_v, n_split).bytes;
    if (!workspace || need == 0 || workspace_bytes < need) return VT_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(workspace) % 256) return VT_ERR_MISALIGNED;
    const vt::Span w{reinterpret_cast<uintptr_t>(workspace), reinterpret_cast<uintptr_t>(workspace) + workspace_bytes};
    const int elt = P.dtype == VT_BF16 ? 2 : 4;
    vt::Span sq, sk, sv, so;  // valid: check_args has passed
    if (!vt::span_of(P.Q, P.qs, P.B, P.H, P.S_q, P.D_qk, elt, &sq) ||
        !vt::span_of(P.K, P.ks, P.B, P.H_kv, P.S_k, P.D_qk, elt, &sk) ||
        !vt::span_of(P.V, P.vs, P.B, P.H_kv, P.S_k, P.D_v, elt, &sv) ||
        !vt::span_of(P.O, P.os, P.B, P.H, P.S_q, P.D_v, elt, &so))
        return VT_ERR_INVALID_ARG;
    if (vt::overlap(w, sq) || vt::overlap(w, sk) || vt::overlap(w, sv) || vt::overlap(w, so)) return VT_ERR_INVALID_ARG;
    if (P.lse) {
        vt::Span sl;
        if (!vt::lse_span(P.lse, P.B, P.H, P.S_q, &sl) || vt::overlap(w, sl)) return VT_ERR_INVALID_ARG;
    }
    return VT_OK;
}

vt_status forward(const Problem &P, const vt_attn_opts *opts, int n_split, void *workspace, cudaStream_t s) {
    const vt_status r = P.dtype == VT_BF16 ? launch<kBF16>(P, opts, n_split, workspace, s)
                                           : launch<kF32>(P, opts, n_split, workspace, s);
    if (r != VT_OK) return r;
    return env_check() ? read_status(s) : VT_OK;
}

// The problem of the entry points that predate the general form: H_kv = H, no lse, causal or not.
Problem plain_problem(const void *Q, const int64_t qs[3], const void *K, const int64_t ks[3], const void *V,
                      const int64_t vs[3], void *O, const int64_t os[3], int64_t B, int64_t H, int64_t S_q,
                      int64_t S_k, int64_t D_qk, int64_t D_v, float scale, int causal, vt_dtype dtype) {
    Problem P{};
    P.Q = Q; P.K = K; P.V = V; P.O = O;
    P.qs = qs; P.ks = ks; P.vs = vs; P.os = os;
    P.lse = nullptr;
    P.B = B; P.H = H; P.H_kv = H > 0 ? H : 1; P.S_q = S_q; P.S_k = S_k; P.D_qk = D_qk; P.D_v = D_v;
    P.scale = scale;
    P.dtype = dtype;
    P.mask = causal ? VT_MASK_CAUSAL : VT_MASK_NONE;
    P.offset = 0;
    P.window = 0;
    return P;
}

}  // namespace
}  // namespace vt

extern "C" {

vt_status vt_attn_fwd_ex(const void *Q, const int64_t q_stride[3], const void *K, const int64_t k_stride[3],
                         const void *V, const int64_t v_stride[3], void *O, const int64_t o_stride[3], int64_t B,
                         int64_t H, int64_t S_q, int64_t S_k, int64_t D_qk, int64_t D_v, float scale, int causal,
                         vt_dtype dtype, const vt_attn_opts *opts, vt_stream_t stream) {
    const vt::NvtxRange range("vt_attn_fwd_ex");
    const vt::Problem P = vt::plain_problem(Q, q_stride, K, k_stride, V, v_stride, O, o_stride, B, H, S_q, S_k, D_qk,
                                            D_v, scale, causal, dtype);
    bool empty = false;
    const vt_status c = vt::check_args(P, &empty);
    if (c != VT_OK || empty) return c;
    return vt::forward(P, opts, 1, nullptr, reinterpret_cast<cudaStream_t>(stream));
}

vt_status vt_attn_fwd_general(const void *Q, const int64_t q_stride[3], const void *K, const int64_t k_stride[3],
                              const void *V, const int64_t v_stride[3], void *O, const int64_t o_stride[3],
                              float *lse, int64_t B, int64_t H, int64_t H_kv, int64_t S_q, int64_t S_k, int64_t D_qk,
                              int64_t D_v, float scale, vt_dtype dtype, const vt_attn_mask *mask, int n_split,
                              void *workspace, size_t workspace_bytes, const vt_attn_opts *opts,
                              vt_stream_t stream) {
    const vt::NvtxRange range("vt_attn_fwd_general");
    vt::Problem P = vt::plain_problem(Q, q_stride, K, k_stride, V, v_stride, O, o_stride, B, H, S_q, S_k, D_qk, D_v,
                                      scale, 0, dtype);
    P.H_kv = H_kv;
    P.lse = lse;
    if (mask) {
        if (mask->reserved != 0) return VT_ERR_INVALID_ARG;
        P.mask = mask->kind;
        P.offset = mask->offset;
        P.window = mask->window;
    }
    bool empty = false;
    const vt_status c = vt::check_args(P, &empty);
    if (c != VT_OK) return c;
    if (n_split < 1) return VT_ERR_INVALID_ARG;
    if (n_split > vt::kMaxSplit) return VT_ERR_UNSUPPORTED;
    if (empty) return VT_OK;
    if (n_split > 1) {
        const vt_status w = vt::check_workspace(P, n_split, workspace, workspace_bytes);
        if (w != VT_OK) return w;
    }
    return vt::forward(P, opts, n_split, workspace, reinterpret_cast<cudaStream_t>(stream));
}

size_t vt_attn_splitkv_workspace_size(int64_t B, int64_t H, int64_t S_q, int64_t D_v, int n_split) {
    if (B <= 0 || H <= 0 || S_q <= 0 || D_v <= 0 || n_split <= 1) return 0;
    return vt::split_layout(B, H, S_q, D_v, n_split).bytes;
}

int vt_attn_splitkv_choose(int64_t B, int64_t H, int64_t S_q, int64_t S_k, int causal, vt_dtype dtype) {
    (void)causal;
    if ((dtype != VT_BF16 && dtype != VT_F32) || B <= 0 || H <= 0 || S_q <= 0 || S_k <= 0) return 1;
    // fp32: the plain call already spreads a unit's key tiles over the CTAs of a cluster
    if (dtype == VT_F32) return 1;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 1;
    // Shares only pay when every CTA still fits in one wave, and each share keeps >= 4 key tiles.
    // work items and key tiles of the kernel that serves the dtype
    const long long rows = vt::q2::kRows;
    const long long bn = vt::q2::kBN;
    const long long items = B * H * ((S_q + rows - 1) / rows);
    const long long tiles = (S_k + bn - 1) / bn;
    long long n = items >= sms ? 1 : sms / items;
    if (n > tiles / 4) n = tiles / 4;
    if (n > vt::kMaxSplit) n = vt::kMaxSplit;
    return n < 1 ? 1 : static_cast<int>(n);
}

vt_status vt_attn_fwd_splitkv(const void *Q, const int64_t q_stride[3], const void *K, const int64_t k_stride[3],
                              const void *V, const int64_t v_stride[3], void *O, const int64_t o_stride[3], int64_t B,
                              int64_t H, int64_t S_q, int64_t S_k, int64_t D_qk, int64_t D_v, float scale, int causal,
                              vt_dtype dtype, int n_split, void *workspace, size_t workspace_bytes,
                              vt_stream_t stream) {
    const vt::NvtxRange range("vt_attn_fwd_splitkv");
    const vt::Problem P = vt::plain_problem(Q, q_stride, K, k_stride, V, v_stride, O, o_stride, B, H, S_q, S_k, D_qk,
                                            D_v, scale, causal, dtype);
    bool empty = false;
    const vt_status c = vt::check_args(P, &empty);
    if (c != VT_OK) return c;
    if (n_split < 1) return VT_ERR_INVALID_ARG;
    if (n_split > vt::kMaxSplit) return VT_ERR_UNSUPPORTED;
    if (empty) return VT_OK;
    if (n_split > 1) {
        const vt_status w = vt::check_workspace(P, n_split, workspace, workspace_bytes);
        if (w != VT_OK) return w;
    }
    return vt::forward(P, nullptr, n_split, workspace, reinterpret_cast<cudaStream_t>(stream));
}

vt_status vt_attn_fwd_splitkv_noalloc(const void *Q, const int64_t q_stride[3], const void *K,
                                      const int64_t k_stride[3], const void *V, const int64_t v_stride[3], void *O,
                                      const int64_t o_stride[3], int64_t B, int64_t H, int64_t S_q, int64_t S_k,
                                      int64_t D_qk, int64_t D_v, float scale, int causal, vt_dtype dtype, int n_split,
                                      vt_stream_t stream) {
    const vt::NvtxRange range("vt_attn_fwd_splitkv_noalloc");
    const vt::Problem P = vt::plain_problem(Q, q_stride, K, k_stride, V, v_stride, O, o_stride, B, H, S_q, S_k, D_qk,
                                            D_v, scale, causal, dtype);
    bool empty = false;
    const vt_status c = vt::check_args(P, &empty);
    if (c != VT_OK) return c;
    if (n_split < 1) return VT_ERR_INVALID_ARG;
    if (n_split > vt::kMaxSplit) return VT_ERR_UNSUPPORTED;
    if (empty) return VT_OK;
    void *scratch = nullptr;
    if (n_split > 1) {
        // The shares' partial results must fit the fixed array; nothing is allocated instead.
        const size_t need = vt::split_layout(B, H, S_q, D_v, n_split).bytes;
        if (need == 0 || need > vt::kNoAllocScratchBytes) return VT_ERR_UNSUPPORTED;
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess) return VT_ERR_CUDA;
        scratch = vt::noalloc_scratch(dev);
        if (!scratch) return VT_ERR_CUDA;
    }
    return vt::forward(P, nullptr, n_split, scratch, reinterpret_cast<cudaStream_t>(stream));
}

vt_status vt_attn_fwd_strided(const void *Q, const int64_t q_stride[3], const void *K, const int64_t k_stride[3],
                              const void *V, const int64_t v_stride[3], void *O, const int64_t o_stride[3], int64_t B,
                              int64_t H, int64_t S_q, int64_t S_k, int64_t D_qk, int64_t D_v, float scale, int causal,
                              vt_dtype dtype, vt_stream_t stream) {
    const vt::NvtxRange range("vt_attn_fwd_strided");
    return vt_attn_fwd_ex(Q, q_stride, K, k_stride, V, v_stride, O, o_stride, B, H, S_q, S_k, D_qk, D_v, scale,
                          causal, dtype, nullptr, stream);
}

vt_status vt_attn_fwd(const void *Q, const void *K, const void *V, void *O, int64_t B, int64_t H, int64_t S_q,
                      int64_t S_k, int64_t D_qk, int64_t D_v, float scale, int causal, vt_dtype dtype,
                      vt_stream_t stream) {
    const vt::NvtxRange range("vt_attn_fwd");
    // Packed strides, formed only from extents that passed the shape checks and only when the products
    // fit in 64 bits: a packed tensor whose element count overflows cannot exist.
    const int64_t unit[3] = {1, 1, 1};
    vt::Problem P = vt::plain_problem(Q, unit, K, unit, V, unit, O, unit, B, H, S_q, S_k, D_qk, D_v, scale, causal,
                                      dtype);
    bool empty = false;
    const vt_status c = vt::check_shape(P, &empty);
    if (c != VT_OK || empty) return c;
    auto packed = [](int64_t H_, int64_t S, int64_t D, int64_t out[3]) {
        out[2] = D;
        return !__builtin_mul_overflow(S, D, &out[1]) && !__builtin_mul_overflow(H_, out[1], &out[0]);
    };
    int64_t qs[3], ks[3], vs[3], os[3];
    if (!packed(H, S_q, D_qk, qs) || !packed(H, S_k, D_qk, ks) || !packed(H, S_k, D_v, vs) || !packed(H, S_q, D_v, os))
        return VT_ERR_INVALID_ARG;
    return vt_attn_fwd_ex(Q, qs, K, ks, V, vs, O, os, B, H, S_q, S_k, D_qk, D_v, scale, causal, dtype, nullptr,
                          stream);
}

}  // extern "C"
