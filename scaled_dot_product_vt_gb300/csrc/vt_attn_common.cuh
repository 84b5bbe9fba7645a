// Definitions shared by the attention kernels: launch parameters, device status bits,
// the per-CTA control block and the time-bounded mbarrier waits.
#pragma once

#include <cuda.h>
#include <cstdint>

#include "vt_ptx.cuh"

namespace vt {

constexpr int kBM = 128;           // query rows per work item (= TMEM lanes)
constexpr int kMaxSplit = 64;       // split-KV shares per work item, at most

constexpr long long kBandInf = 1LL << 42;  // a band edge that no row reaches

// Device status bits (the host maps them to vt_status codes).
constexpr unsigned kStatusTimeout = 1u;
constexpr unsigned kStatusBounds = 2u;

enum : int { kF32 = 0, kBF16 = 1 };

struct AttnParams {
    int B, H, S_q, S_k, D_qk, D_v;
    int n_qblocks;    // query blocks per (b, h): ceil(S_q / rows per block)
    int n_units;      // work units of a launch: query blocks x heads x batches x n_split
    int head_group;   // heads whose query blocks are interleaved in the launch order
    int qk_ksteps;    // ceil(D_qk / K-step), K-step = 16 (bf16) or 8 (tf32)
    int q_chunks;     // 128-byte column chunks of a Q/K row: ceil(D_qk * elt / 128)
    int v_chunks;     // 128-byte column chunks of a V row
    int n_pv;         // MMA N of P*V: D_v rounded up to 16
    int stages;
    // Allowed keys of query row i: [i + band_lo, i + band_hi] within [0, S_k); +-kBandInf stands
    // for "no limit" (the host maps each mask kind to its band).
    long long band_lo, band_hi;
    int reverse_q;     // 1: launch the query blocks last-first (work grows with the block index)
    int kv_group;      // query heads per key/value head: K/V head of query head h is h / kv_group
    float scale_log2;  // scale * log2(e)
    float *lse;        // nullptr, or [B*H*S_q] natural-log log-sum-exp per row
    void *O;
    long long o_sb, o_sh, o_ss;  // element strides of O for b, h, s
    int o_vec32;                 // 1: O and its strides are 32-byte multiples (32-byte stores of O rows)
    const void *V;               // read by the fp32 V loader
    long long v_sb, v_sh, v_ss;
    const void *Q;               // read by the fp32 kernel's softmax threads (Q goes to TMEM)
    long long q_sb, q_sh, q_ss;
    // fp32 kernel: query tiles per work unit (1 or 2), and the CTAs of a thread-block cluster that share
    // one unit's key tiles and merge their results in distributed shared memory (1: no cluster)
    int tiles_per_unit;
    int cluster;
    // Split-KV: each work item's key tiles are cut into n_split contiguous ranges, one per CTA; with
    // n_split > 1 the CTAs write unnormalised partial outputs (fp32, D_v per row), their row max m
    // (log2 units, -inf if no allowed key), row sum l and the correction that makes l + corr weigh P
    // as the bf16 values P V used, indexed [split][(b*H + h)*S_q + i].
    int n_split;
    float *part_o;
    float *part_m;
    float *part_l;
    float *part_c;
    unsigned long long timeout_ns;
    unsigned flags;
    unsigned *status;  // device status word of the launching stream
};

// First allowed key of row r and one past its last, clamped to [0, S_k] (empty when lo >= hi).
__device__ __forceinline__ int band_key_lo(const AttnParams &p, int r) {
    const long long x = static_cast<long long>(r) + p.band_lo;
    return static_cast<int>(x < 0 ? 0 : (x > p.S_k ? p.S_k : x));
}
__device__ __forceinline__ int band_key_hi(const AttnParams &p, int r) {
    const long long x = static_cast<long long>(r) + p.band_hi + 1;
    return static_cast<int>(x < 0 ? 0 : (x > p.S_k ? p.S_k : x));
}

// Key tiles [*a, *e) of `bn` keys that query rows first..last need (an empty range as 0, 0).
__device__ __forceinline__ void band_tiles(const AttnParams &p, int first, int last, int bn, int *a, int *e) {
    const int lo = band_key_lo(p, first), hi = band_key_hi(p, last);
    if (lo < hi) {
        *a = lo / bn;
        *e = (hi + bn - 1) / bn;
    } else {
        *a = 0;
        *e = 0;
    }
}

// log(sum of exponentials) in natural-log units from a log2-unit reference max m and sum l.
__device__ __forceinline__ float lse_from(float m, float l) {
    return l > 0.0f ? (m + log2f(l)) * 0.69314718055994531f : -INFINITY;
}

// Device index checks of the debug build (-DVT_DEBUG): a failed check records the bounds bit of the
// status word and the CTA's abort flag, and the caller skips the access it guards and stops.  Release
// builds compile the checks out (the condition is not evaluated).
#ifdef VT_DEBUG
#define VT_DEV_CHECK(cond, abort_flag, p) ::vt::dev_check((cond), (abort_flag), (p))
#else
#define VT_DEV_CHECK(cond, abort_flag, p) true
#endif
constexpr unsigned kFlagTestStall = 1u;   // VT_OPT_TEST_STALL
constexpr unsigned kFlagTestBounds = 2u;  // VT_OPT_TEST_BOUNDS (debug build)

__device__ __forceinline__ bool dev_check(bool ok, volatile uint32_t &abort_flag, const AttnParams &p) {
    if (!ok) {
        abort_flag = 1;
        atomicOr(p.status, kStatusBounds);
    }
    return ok;
}

// Wait for the phase of `bar` with `parity`, giving up after the time limit or when
// another role has aborted.  Returns false on give-up (after flagging the abort).
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, volatile uint32_t &abort_flag,
                                             const AttnParams &p) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t n = 1;; ++n) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((n & 63u) == 0) {
            if (abort_flag) return false;
            if (globaltimer_ns() - t0 > p.timeout_ns) {
                abort_flag = 1;
                atomicOr(p.status, kStatusTimeout);
                return false;
            }
        }
    }
}

// Wait until a shared-memory counter exceeds `above`, with the same time limit and abort shortcut as
// wait_bounded.
__device__ __forceinline__ bool wait_flag_above(volatile uint32_t &flag, int above, volatile uint32_t &abort_flag,
                                                const AttnParams &p) {
    if (static_cast<int>(flag) > above) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t n = 1;; ++n) {
        if (static_cast<int>(flag) > above) return true;
        if ((n & 63u) == 0) {
            if (abort_flag) return false;
            if (globaltimer_ns() - t0 > p.timeout_ns) {
                abort_flag = 1;
                atomicOr(p.status, kStatusTimeout);
                return false;
            }
        }
    }
}

// Wait without the abort shortcut (used while draining copies in flight on the abort path).
__device__ __forceinline__ void wait_drain(uint32_t bar, uint32_t parity, const AttnParams &p) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > p.timeout_ns) {
            atomicOr(p.status, kStatusTimeout);
            return;
        }
    }
}

}  // namespace vt
