// Definitions shared by the attention kernels: launch parameters, device status bits,
// the per-CTA control block and the time-bounded mbarrier waits.
#pragma once

#include <cuda.h>
#include <cstdint>

#include "vt_ptx.cuh"

namespace vt {

constexpr int kBM = 128;           // query rows per work item (= TMEM lanes)
constexpr int kMaxStages = 4;
constexpr int kMaxSplit = 64;       // split-KV shares per work item, at most
constexpr float kRescaleTau = 8.0f;  // log2 units: rescale O only when the row max grows by more

// Device status bits (the host maps them to vt_status codes).
constexpr unsigned kStatusTimeout = 1u;
constexpr unsigned kStatusBounds = 2u;

enum : int { kF32 = 0, kBF16 = 1 };

struct AttnParams {
    int B, H, S_q, S_k, D_qk, D_v;
    int n_qblocks;    // query blocks per (b, h): ceil(S_q / rows per CTA)
    int head_group;   // heads whose query blocks are interleaved in the launch order
    int qk_ksteps;    // ceil(D_qk / K-step), K-step = 16 (bf16) or 8 (tf32)
    int q_chunks;     // 128-byte column chunks of a Q/K row: ceil(D_qk * elt / 128)
    int v_chunks;     // 128-byte column chunks of a V row
    int n_pv;         // MMA N of P*V: D_v rounded up to 16
    int stages;
    int causal;
    float scale_log2;  // scale * log2(e)
    void *O;
    long long o_sb, o_sh, o_ss;  // element strides of O for b, h, s
    const void *V;               // read by the fp32 V loader
    long long v_sb, v_sh, v_ss;
    // Split-KV: each work item's key tiles are cut into n_split contiguous ranges, one per CTA; with
    // n_split > 1 the CTAs write unnormalised partial outputs (fp32, D_v per row), their row max m
    // (log2 units, -inf if no allowed key) and row sum l, indexed [split][(b*H + h)*S_q + i].
    int n_split;
    float *part_o;
    float *part_m;
    float *part_l;
    unsigned long long timeout_ns;
    unsigned flags;
    unsigned *status;  // device status word
};


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
