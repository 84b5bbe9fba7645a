// Split-KV merge: combine the per-share partial outputs of one query row into O.
//
// Share s of row r holds an unnormalised output O_s (fp32, D_v values), its reference max m_s
// (log2 units; -inf when the share had no allowed key) and its sum l_s, all relative to m_s.  In
// real arithmetic O[r] = sum_s 2^(m_s - M) O_s / sum_s 2^(m_s - M) l_s for any M; M = max_s m_s
// keeps every weight <= 1.  This is the continuation step of the coverage table's
// attention_fwd_triton3 row (case 4 reads M, L and Out and merges a further key range), applied
// to all shares at once.  HBM-bound: per row it reads n_split * (D_v + 3) floats (O, m, l and the correction) and writes D_v.
// The row's log-sum-exp, if asked for, is M + log2(L) in natural-log units.
#pragma once

#include <cstdint>

#include "vt_attn_common.cuh"

namespace vt {

struct MergeParams {
    const float *part_o;
    const float *part_m;
    const float *part_l;
    const float *part_c;
    void *O;
    float *lse;      // nullptr, or one natural-log log-sum-exp per row
    long long rows;  // B * H * S_q
    int H, S_q, D_v, n_split;
    long long o_sb, o_sh, o_ss;
};

constexpr int kMergeRowsPerBlock = 4;  // one warp per row

// ELT: 2 = bf16 output, 4 = fp32 output.  D_v <= 128: lane L handles columns L, L+32, L+64, L+96.
template <int ELT>
__global__ void __launch_bounds__(32 * kMergeRowsPerBlock)
    attn_merge_kernel(const MergeParams mp) {
    const int lane = threadIdx.x & 31;
    const long long row = static_cast<long long>(blockIdx.x) * kMergeRowsPerBlock + (threadIdx.x >> 5);
    if (row >= mp.rows) return;
    // One pass over the shares in groups of four: a group's m, l, correction and O values are all loaded
    // before any is used (one memory round trip per group), and the running sums are rescaled when the
    // running max M grows:  M' = max(M, m_s),  sums *= 2^(M - M'),  then each share adds 2^(m_s - M') times its own.
    float M = -INFINITY;
    float L = 0.0f;   // sum of the shares' l: the log-sum-exp
    float Lo = 0.0f;  // sum of l + corr: the divisor of O, weighing P as P V used it
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int s0 = 0; s0 < mp.n_split; s0 += 4) {
        float ms[4], ls[4], cs[4], o[4][4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const bool in = s0 + u < mp.n_split;
            const long long idx = static_cast<long long>(s0 + u) * mp.rows + row;
            ms[u] = in ? mp.part_m[idx] : -INFINITY;
            ls[u] = in ? mp.part_l[idx] : 0.0f;
            cs[u] = in ? mp.part_c[idx] : 0.0f;
            const float *po = mp.part_o + idx * mp.D_v;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int col = lane + 32 * c;
                o[u][c] = (in && col < mp.D_v) ? po[col] : 0.0f;
            }
        }
        const float Mn = fmaxf(fmaxf(M, fmaxf(ms[0], ms[1])), fmaxf(ms[2], ms[3]));
        if (Mn == -INFINITY) continue;  // no allowed key in any share so far
        const float r = M == -INFINITY ? 0.0f : ex2(M - Mn);
        L *= r;
        Lo *= r;
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[c] *= r;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            if (ms[u] == -INFINITY) continue;  // no allowed key in this share (or no share)
            const float w = ex2(ms[u] - Mn);
            L += w * ls[u];
            Lo += w * (ls[u] + cs[u]);
#pragma unroll
            for (int c = 0; c < 4; ++c) acc[c] += w * o[u][c];
        }
        M = Mn;
    }
    const float inv = L > 0.0f ? 1.0f / Lo : 0.0f;  // no share saw an allowed key: the row is 0
    if (mp.lse && lane == 0) mp.lse[row] = lse_from(M, L);
    const long long i = row % mp.S_q;
    const long long bh = row / mp.S_q;
    const long long h = bh % mp.H, b = bh / mp.H;
    uint8_t *orow = reinterpret_cast<uint8_t *>(mp.O) + (b * mp.o_sb + h * mp.o_sh + i * mp.o_ss) * ELT;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const int col = lane + 32 * c;
        if (col >= mp.D_v) continue;
        const float v = acc[c] * inv;
        if (ELT == 2) {
            reinterpret_cast<uint16_t *>(orow)[col] = static_cast<uint16_t>(pack_bf16x2(v, 0.0f) & 0xFFFFu);
        } else {
            reinterpret_cast<float *>(orow)[col] = v;
        }
    }
}

}  // namespace vt
