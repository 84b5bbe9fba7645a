// Attention forward, fp32 I/O on the TF32 tensor path, for sm_103a.
//
// A work unit is one or two 128-row query tiles of one (b, h) slice that share every 64-key K/V tile,
// and one share of their key tiles.  With two tiles, the tensor core works for one tile while the other
// tile's softmax warpgroup computes (the same ping-pong as the bf16 kernel).  The shares of a unit either
// run as the CTAs of one thread-block cluster, which merge their partial results through distributed
// shared memory at the end (no second launch, no global scratch), or, with a caller workspace
// (vt_attn_fwd_splitkv), as separate CTAs that write partial results for the merge kernel.
//
// TF32 specifics.  Q is held in TMEM and is the A operand of S = Q K^T (the TS form runs at the full
// tensor rate for 64-key tiles, the shared-memory form at two thirds), so shared memory holds only the
// K/V ring.  kind::tf32 reads its B operand K-major only, so V tiles, which TMA brings in as they are
// stored (d contiguous), are transposed inside shared memory (keys contiguous) by transposer warps.
// Q tiles come by TMA too, into the memory of the ring's last stages, and each softmax thread copies its row
// into TMEM.  Latency: the Q tiles and the first stages' K and V are requested before the CTA's set-up
// barrier, so their memory latency overlaps the barrier and TMEM set-up.
//
// Warp roles (16 warps):
//   warp 0              TMA producer: K_j and V_j into stage j of a ring of stages
//   warps 1 / 13        MMA issuers of query tiles 0 / 1 (warp 1 also owns TMEM); each whole warp runs the
//                       issuing code with warp-uniform values and one lane, elected once, issues.  Per key tile j
//                       of its range:  O_t += P_t,j V_j,  S_t = Q_t K_{j+1}^T
//   warps 4-7 / 8-11    softmax warpgroups of query tiles 0 / 1, one row per thread: each first copies its
//                       row of Q from shared memory into TMEM, then runs the online softmax and the epilogue
//   warps 2, 3, 12, 14, 15  V transposers: V_j read from its TMA staging area with 16-byte loads and
//                       written transposed (V^T, keys contiguous, 128-byte swizzle) into the V^T area of
//                       stage j
// TMEM columns: S_t (64 each), then O_t (n_pv each), then Q_t (D_qk rounded up to 8 each).  P_t,j
// overwrites S_t,j as fp32 values and is the A operand of O_t += P_t,j V_j.
//
// The decomposition (query block, head, batch), the tail masks and the write set follow the FA-1
// boundary kernel verified on the VeriTile page "VeriTile.Examples.FlashAttention1.NaiveRefinement";
// the reductions are the accy page's score_dot, score_max, score_exp_sum and value_weighted_sum,
// computed online with the base-2 exponential of the folded scale; the cluster merge is the
// continuation step of the VeriTile coverage table's attention_fwd_triton3 row (case 4: an output,
// its max and its sum merged with those of further keys).
#pragma once

#include <cuda.h>
#include <cstdint>

#include "vt_attn_common.cuh"

namespace vt {
namespace f2 {

constexpr int kBN = 64;             // keys per tile
constexpr int kThreads = 512;       // 16 warps
constexpr int kMaxStages = 6;  // 4 barriers per stage, one per lane of warp 0 (lanes 24-31 take the rest)
constexpr int kLoaderThreads = 160;  // V transposers: warps 2, 3, 12, 14, 15
constexpr int kMaxVItems = 4;        // 4-key x 4-column blocks of V per transposer thread and tile, at most
constexpr float kTau = 8.0f;         // lazy-rescale threshold (log2 units)
constexpr int kMaxCluster = 8;

struct Ctl {
    uint64_t full_k[kMaxStages];
    uint64_t full_vs[kMaxStages];  // V_j landed in the staging area (TMA)
    uint64_t full_v[kMaxStages];   // V_j^T written (transposer arrivals)
    uint64_t empty[kMaxStages];
    uint64_t q_smem;      // Q tiles landed in shared memory (TMA)
    uint64_t q_full[2];   // Q_t in TMEM (128 arrivals); also: the thread no longer reads Q from shared memory
    uint64_t s_full[2];   // scores of tile t ready (and every earlier MMA done)
    uint64_t p_full[2];   // P of tile t written (128 arrivals)
    uint64_t o_done[2];   // last P V of tile t done
    uint64_t drain[2];  // a stopping MMA warp's products are done (one per MMA warp)
    uint64_t recv_full;  // cluster merge: the other CTAs' partial rows for this CTA's rows have landed
    uint64_t stall;
    uint32_t tmem_base;
    volatile uint32_t abort_flag;
    volatile uint32_t t0_issued;  // key tiles whose products MMA warp 1 (tile 0) has issued
};

// Index of a transposer thread (0 .. kLoaderThreads - 1), or -1 for the other warps.
__device__ __forceinline__ int loader_index(int warp, int lane) {
    const int w = warp == 2 ? 0 : warp == 3 ? 1 : warp == 12 ? 2 : warp == 14 ? 3 : warp == 15 ? 4 : -1;
    return w < 0 ? -1 : w * 32 + lane;
}

// One unit of a CTA: its (b, h, K/V head, first row), its share of the key tiles [j0, j0 + n_kv) and,
// per query tile t, the tiles [as_t, es_t) of the share that the tile needs (relative to j0).
struct Unit {
    int b, h, hk, r0, share;
    int j0, n_kv;
    int as[2], es[2];
};

// Units run all heads' heaviest query blocks first when work grows with the block index; the shares of
// one unit are adjacent CTAs (one cluster when the shares merge in distributed shared memory).
__device__ __forceinline__ Unit decode(const AttnParams &p, int cta) {
    Unit U;
    const int n_share = p.cluster > 1 ? p.cluster : p.n_split;
    U.share = cta % n_share;
    const int item = cta / n_share;
    const int bh_count = p.B * p.H;
    const int slot = item / bh_count;
    const int bh = item - slot * bh_count;
    const int qb = p.reverse_q ? (p.n_qblocks - 1 - slot) : slot;
    U.h = bh % p.H;
    U.b = bh / p.H;
    U.hk = U.h / p.kv_group;
    U.r0 = qb * kBM * p.tiles_per_unit;
    int a[2] = {0, 0}, e[2] = {0, 0};
    for (int t = 0; t < p.tiles_per_unit; ++t) {
        const int first = U.r0 + t * kBM;
        if (first < p.S_q) band_tiles(p, first, min(first + kBM, p.S_q) - 1, kBN, &a[t], &e[t]);
    }
    const bool has0 = e[0] > a[0], has1 = e[1] > a[1];
    const int A = has0 ? (has1 ? min(a[0], a[1]) : a[0]) : (has1 ? a[1] : 0);
    const int E = has0 ? (has1 ? max(e[0], e[1]) : e[0]) : (has1 ? e[1] : 0);
    const int n_item = E - A;
    const int per = (n_item + n_share - 1) / n_share;
    const int lo = min(U.share * per, n_item), hi = min(n_item, lo + per);
    U.j0 = A + lo;
    U.n_kv = hi - lo;
    for (int t = 0; t < 2; ++t) {
        U.as[t] = min(max(a[t] - U.j0, 0), U.n_kv);
        U.es[t] = min(max(e[t] - U.j0, 0), U.n_kv);
        if (U.es[t] <= U.as[t]) U.as[t] = U.es[t] = 0;
    }
    return U;
}

// Invariants of a decoded unit, checked by the debug build before any load of the unit.
__device__ __forceinline__ bool unit_valid(const AttnParams &p, const Unit &U) {
    const int tiles = (p.S_k + kBN - 1) / kBN;
    return U.b >= 0 && U.b < p.B && U.h >= 0 && U.h < p.H && U.hk == U.h / p.kv_group && U.r0 >= 0 &&
           U.r0 < p.S_q && U.j0 >= 0 && U.n_kv >= 0 && U.j0 + U.n_kv <= tiles && U.as[0] >= 0 &&
           U.as[0] <= U.es[0] && U.es[0] <= U.n_kv && U.as[1] >= 0 && U.as[1] <= U.es[1] && U.es[1] <= U.n_kv;
}

}  // namespace f2

// KQ: the most MMA K-steps (8 tf32 each) of Q K^T the instantiation runs (D_qk rounded up to 8, then to
// 32, 64, 96 or 128); the steps past D_qk are skipped.
template <int KQ, bool FOLD>
__global__ void __launch_bounds__(f2::kThreads, 1)
    attn_fwd_f32_2q_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                           const __grid_constant__ CUtensorMap tmV, const AttnParams p) {
    using namespace f2;
    constexpr int BN = kBN;
    __shared__ Ctl ctl;
    extern __shared__ uint8_t smem_raw[];

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int T = p.tiles_per_unit;
    const Unit U = decode(p, blockIdx.x);
    const int n_kv = U.n_kv;

    // shared memory: `stages` stages of (K tile, V tile as loaded, V^T tile), 1024-byte aligned for the
    // 128-byte swizzle
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const uint32_t k_bytes = p.q_chunks * BN * 128;
    const uint32_t vs_bytes = p.v_chunks * BN * 128;
    const uint32_t v_bytes = p.n_pv * BN * 4;
    const uint32_t stage_bytes = k_bytes + vs_bytes + v_bytes;
    auto sK = [&](int st) { return base + st * stage_bytes; };
    auto sVs = [&](int st) { return base + st * stage_bytes + k_bytes; };
    auto sV = [&](int st) { return base + st * stage_bytes + k_bytes + vs_bytes; };
    // The Q tiles arrive by TMA in the memory of the ring's last q_stages stages, which take K and V only
    // once every tile's Q is in TMEM.
    const uint32_t q_tile_bytes = p.q_chunks * kBM * 128;
    const int q_stages = static_cast<int>((T * q_tile_bytes + stage_bytes - 1) / stage_bytes);
    const uint32_t sQ = base + (p.stages - q_stages) * stage_bytes;
    const int dq = p.qk_ksteps * 8;  // TMEM columns of one Q tile
    const uint32_t col_s0 = 0, col_o0 = static_cast<uint32_t>(BN * T);
    const uint32_t col_q0 = col_o0 + static_cast<uint32_t>(T * p.n_pv);

#ifdef VT_DEBUG
    const bool unit_valid_here = !(p.flags & kFlagTestBounds) && unit_valid(p, U);
#else
    const bool unit_valid_here = true;  // the release build evaluates no device check
#endif
    const bool is_softmax = warp >= 4 && warp < 12;
    const int t = is_softmax ? (warp - 4) >> 2 : 0;
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const int q_row = U.r0 + t * kBM + row;
    const int n_my = U.es[t] - U.as[t];

    // Barriers are initialised by warp 0; thread 0 then issues the first stages' K and V loads before the
    // set-up barrier.
    int issued = 0;  // K/V stages the producer has loaded
    if (warp == 0) {
        // one barrier per lane: stage s of full_k / full_vs / full_v / empty is barrier 4 s + k
        if (lane < 4 * p.stages) {
            const int st = lane >> 2, k = lane & 3;
            uint64_t *bar = k == 0 ? &ctl.full_k[st] : k == 1 ? &ctl.full_vs[st] : k == 2 ? &ctl.full_v[st] : &ctl.empty[st];
            mbar_init(smem_u32(bar), k == 2 ? kLoaderThreads : k == 3 ? 2 : 1);  // empty: one arrival per MMA warp
        } else if (lane >= 24) {
            const int i = lane - 24;  // 8 barriers: q_full, s_full, p_full, o_done of the two tiles
            uint64_t *bar = (i >> 1) == 0 ? &ctl.q_full[i & 1] : (i >> 1) == 1 ? &ctl.s_full[i & 1]
                            : (i >> 1) == 2 ? &ctl.p_full[i & 1] : &ctl.o_done[i & 1];
            mbar_init(smem_u32(bar), ((i >> 1) == 0 || (i >> 1) == 2) ? 128 : 1);
        }
        if (lane == 0) {
            mbar_init(smem_u32(&ctl.drain[0]), 1);
            mbar_init(smem_u32(&ctl.drain[1]), 1);
            mbar_init(smem_u32(&ctl.recv_full), 1);
            mbar_init(smem_u32(&ctl.q_smem), 1);
            mbar_init(smem_u32(&ctl.stall), 1);
            ctl.abort_flag = 0;
            ctl.t0_issued = 0;
        }
        fence_mbar_init();  // each lane's initialisations, for the TMA loads thread 0 issues next
        __syncwarp();
    }
    if (threadIdx.x == 0) {
        if (unit_valid_here) {
            tma_prefetch_desc(&tmQ);
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmV);
            if (n_kv > 0) {
                const bool q0 = U.es[0] > U.as[0], q1 = T > 1 && U.es[1] > U.as[1];  // tiles with work need Q
                mbar_arrive_expect_tx(smem_u32(&ctl.q_smem), (int(q0) + int(q1)) * q_tile_bytes);
                for (int tt = 0; tt < 2; ++tt) {
                    if (!(tt == 0 ? q0 : q1)) continue;
                    for (int c = 0; c < p.q_chunks; ++c)
                        tma_load_4d(sQ + tt * q_tile_bytes + c * kBM * 128, &tmQ, smem_u32(&ctl.q_smem), c * 32,
                                    U.r0 + tt * kBM, U.h, U.b);
                }
            }
            for (; issued < n_kv && issued < p.stages - q_stages; ++issued) {
                const int st = issued, key0 = (U.j0 + issued) * BN;
                mbar_arrive_expect_tx(smem_u32(&ctl.full_k[st]), k_bytes);
                for (int c = 0; c < p.q_chunks; ++c)
                    tma_load_4d(sK(st) + c * BN * 128, &tmK, smem_u32(&ctl.full_k[st]), c * 32, key0, U.hk, U.b);
                mbar_arrive_expect_tx(smem_u32(&ctl.full_vs[st]), vs_bytes);
                for (int c = 0; c < p.v_chunks; ++c)
                    tma_load_4d(sVs(st) + c * BN * 128, &tmV, smem_u32(&ctl.full_vs[st]), c * 32, key0, U.hk, U.b);
            }
        }
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&ctl.tmem_base), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctl.tmem_base;
    const bool unit_ok = VT_DEV_CHECK(unit_valid_here, ctl.abort_flag, p);

    // per softmax thread: its final statistics (used by the epilogue after the role code)
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
    float m_used = -INFINITY;  // reference max (log2 units) of O_t and l
    float l = 0.0f;
    bool ok = true;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer (K and V tiles)
        if (lane == 0 && n_kv > 0 && unit_ok) {
            const bool q0 = U.es[0] > U.as[0], q1 = T > 1 && U.es[1] > U.as[1];
            for (int j = issued; j < n_kv; ++j) {
                const int st = j % p.stages, use = j / p.stages;
                if (use == 0) {  // a stage of the Q region: its Q must have reached TMEM
                    if (q0 && !wait_bounded(smem_u32(&ctl.q_full[0]), 0, ctl.abort_flag, p)) break;
                    if (q1 && !wait_bounded(smem_u32(&ctl.q_full[1]), 0, ctl.abort_flag, p)) break;
                }
                if (use > 0 && !wait_bounded(smem_u32(&ctl.empty[st]), (use - 1) & 1, ctl.abort_flag, p)) break;
                if (!VT_DEV_CHECK((U.j0 + j) * BN < p.S_k, ctl.abort_flag, p)) break;
                const int key0 = (U.j0 + j) * BN;
                mbar_arrive_expect_tx(smem_u32(&ctl.full_k[st]), k_bytes);
                for (int c = 0; c < p.q_chunks; ++c)
                    tma_load_4d(sK(st) + c * BN * 128, &tmK, smem_u32(&ctl.full_k[st]), c * 32, key0, U.hk, U.b);
                mbar_arrive_expect_tx(smem_u32(&ctl.full_vs[st]), vs_bytes);
                for (int c = 0; c < p.v_chunks; ++c)
                    tma_load_4d(sVs(st) + c * BN * 128, &tmV, smem_u32(&ctl.full_vs[st]), c * 32, key0, U.hk, U.b);
                issued = j + 1;
            }
        }
        if (lane == 0 && ctl.abort_flag) {
            // let every copy this thread started land before the CTA's memory goes away
            if (n_kv > 0 && unit_ok && (U.es[0] > U.as[0] || (T > 1 && U.es[1] > U.as[1])))
                wait_drain(smem_u32(&ctl.q_smem), 0, p);
            for (int j = max(0, issued - p.stages); j < issued; ++j) {
                wait_drain(smem_u32(&ctl.full_k[j % p.stages]), (j / p.stages) & 1, p);
                wait_drain(smem_u32(&ctl.full_vs[j % p.stages]), (j / p.stages) & 1, p);
            }
        }
    } else if (warp == 1 || warp == 13) {
        // ------------------------------------------------------------ MMA issuers, one warp per query tile
        // Warp 1 issues tile 0's products, warp 13 tile 1's, so neither tile's next Q K^T waits behind the
        // other tile's issue.  Both release every stage they were given (empty[] counts two arrivals); a stage
        // outside a tile's key range is released once it has been loaded, which keeps each arrival in the
        // phase of the stage's current use.
        const int tm = warp == 1 ? 0 : 1;
        if (n_kv > 0 && unit_ok) {
            const uint32_t idesc_qk = instr_desc(2, kBM, BN, 0);
            const uint32_t idesc_pv = instr_desc(2, kBM, p.n_pv, 0);
            const uint64_t kdesc0 = smem_desc_sw128(sK(0), 16, 1024);
            const uint64_t vdesc0 = smem_desc_sw128(sV(0), 16, 1024);  // V^T, K-major
            const uint32_t k_lo0 = static_cast<uint32_t>(kdesc0), k_hi = static_cast<uint32_t>(kdesc0 >> 32);
            const uint32_t v_lo0 = static_cast<uint32_t>(vdesc0), v_hi = static_cast<uint32_t>(vdesc0 >> 32);
            const uint32_t stage_step = stage_bytes >> 4;
            const uint32_t v_chunk = static_cast<uint32_t>(p.n_pv) * 8;  // one 32-key chunk of V^T, descriptor units
            const int ksteps = p.qk_ksteps;
            const int as = tm < T ? U.as[tm] : 0, es = tm < T ? U.es[tm] : 0;
            const uint32_t s_col = tmem + col_s0 + tm * BN, o_col = tmem + col_o0 + tm * p.n_pv;
            const uint32_t q_col = tmem + col_q0 + tm * dq;
            bool any_mma = false;
            // The lane that issues every MMA and commit of this warp, elected once (a commit tracks the MMAs of
            // the thread that issues it).  Every lane waits, so the issuing lane has itself observed the phase.
            const uint32_t lead = elect_leader();
            auto wait1 = [&](uint32_t bar, uint32_t parity) -> bool {
                return __all_sync(0xffffffffu, wait_bounded(bar, parity, ctl.abort_flag, p)) != 0;
            };
            // S = Q K_j^T over the ksteps K-steps of D_qk: one jump into an unrolled sequence that runs steps
            // ksteps - 1 down to 0 (the first one issued overwrites, the rest accumulate), so no step carries
            // a test of its own.
            auto qk = [&](int j) {
                const uint32_t k_lo = k_lo0 + (j % p.stages) * stage_step;
                uint32_t acc = 0;
#define VT_QK_STEP(kk)                                                                                             \
    case (kk) + 1:                                                                                                 \
        if ((kk) < KQ) {                                                                                           \
            mma_ts_tf32_lead(s_col, q_col + (kk) * 8, k_lo + ((kk) >> 2) * (BN * 8) + ((kk) & 3) * 2, k_hi,         \
                             idesc_qk, acc, lead);                                                                 \
            acc = 1;                                                                                               \
        }
                switch (ksteps) {
                    VT_QK_STEP(15) VT_QK_STEP(14) VT_QK_STEP(13) VT_QK_STEP(12) VT_QK_STEP(11) VT_QK_STEP(10)
                    VT_QK_STEP(9) VT_QK_STEP(8) VT_QK_STEP(7) VT_QK_STEP(6) VT_QK_STEP(5) VT_QK_STEP(4)
                    VT_QK_STEP(3) VT_QK_STEP(2) VT_QK_STEP(1) VT_QK_STEP(0)
                    default: break;
                }
#undef VT_QK_STEP
                any_mma = true;
            };
            auto pv = [&](int j, uint32_t acc0) {
                const uint32_t v_lo = v_lo0 + (j % p.stages) * stage_step;
#pragma unroll
                for (int kk = 0; kk < BN / 8; ++kk)
                    mma_ts_tf32_lead(o_col, s_col + kk * 8, v_lo + (kk >> 2) * v_chunk + (kk & 3) * 2, v_hi, idesc_pv,
                                     (acc0 | kk) ? 1u : 0u, lead);
            };

            if (p.flags & kFlagTestStall) ok = wait1(smem_u32(&ctl.stall), 0);  // test hook: never signalled
            if (ok && es > as) {
                ok = wait1(smem_u32(&ctl.q_full[tm]), 0);
                tc_fence_after();  // Q was written to TMEM by the softmax warps
                if (ok) ok = wait1(smem_u32(&ctl.full_k[as % p.stages]), (as / p.stages) & 1);
                if (ok) {
                    qk(as);
                    mma_commit_lead(smem_u32(&ctl.s_full[tm]), lead);
                }
            }
            uint32_t p_par = 0;
            for (int j = 0; ok && j < n_kv; ++j) {
                const int st = j % p.stages;
                if (!(ok = wait1(smem_u32(&ctl.full_v[st]), (j / p.stages) & 1))) break;
                if (j >= as && j < es) {
                    if (!(ok = wait1(smem_u32(&ctl.p_full[tm]), p_par))) break;
                    // tile 1's products of key tile j go to the tensor core after tile 0's, so the two tiles keep
                    // half a step apart and each one's softmax overlaps the other's products
                    if (tm == 1 && !(ok = __all_sync(0xffffffffu, wait_flag_above(ctl.t0_issued, j, ctl.abort_flag, p))))
                        break;
                    p_par ^= 1u;
                    tc_fence_after();  // P was written to TMEM and V^T to shared memory by other warps
                    pv(j, j > as);
                    if (j + 1 < es) {
                        if (!(ok = wait1(smem_u32(&ctl.full_k[(j + 1) % p.stages]), ((j + 1) / p.stages) & 1))) break;
                        qk(j + 1);
                        mma_commit_lead(smem_u32(&ctl.s_full[tm]), lead);
                    } else {
                        mma_commit_lead(smem_u32(&ctl.o_done[tm]), lead);
                    }
                }
                mma_commit_lead(smem_u32(&ctl.empty[st]), lead);  // this tile is done with stage st
                if (tm == 0) {
                    __syncwarp();
                    if (lane == 0) ctl.t0_issued = static_cast<uint32_t>(j + 1);
                }
            }
            if (tm == 0 && lane == 0) ctl.t0_issued = 0x7FFFFFFFu;  // stopped or done: never hold tile 1 back
            if (!ok && any_mma) {
                mma_commit_lead(smem_u32(&ctl.drain[tm]), lead);
                if (lane == 0) wait_drain(smem_u32(&ctl.drain[tm]), 0, p);
                __syncwarp();
            }
        }
    } else if (!is_softmax) {
        // ------------------------------------------------------------ V transposers
        const int lt = loader_index(warp, lane);
        if (lt >= 0 && unit_ok) {
            const int nd4 = p.n_pv / 4;  // 4-column groups, including the zero padding up to n_pv
            const int n_items = (BN / 4) * nd4;
            uint8_t *smem_gen = smem_raw + (base - raw);
            for (int j = 0; j < n_kv; ++j) {
                const int st = j % p.stages;
                // the staging area of stage st is reloaded only after the stage's empty phase, which needs this
                // stage's V^T: waiting for its full phase is enough
                bool w = wait_bounded(smem_u32(&ctl.full_vs[st]), (j / p.stages) & 1, ctl.abort_flag, p);
                if (!__all_sync(0xffffffffu, w)) break;
                const uint8_t *src = smem_gen + (sVs(st) - base);
                uint8_t *dst = smem_gen + (sV(st) - base);
                // An item is a block of 4 keys x 4 columns: four 16-byte loads of V rows (key k: 128-byte row k of
                // the column chunk, 16-byte unit swizzled with k mod 8), a register transpose, and four 16-byte
                // stores of 4 consecutive keys of one column (16 contiguous bytes of V^T, kept together by the
                // swizzle).  Items run key-group fastest, so each 8-lane store phase covers 8 different 16-byte
                // units of one V^T row.  Columns past D_v are zero (TMA fills them) and keys past S_k too.
                float4 blk[kMaxVItems][4];
#pragma unroll
                for (int u = 0; u < kMaxVItems; ++u) {
                    const int item = lt + u * kLoaderThreads;
                    const int kg = item % (BN / 4);
                    const int d0 = (item / (BN / 4)) * 4;
                    const int ch = d0 >> 5, unit = (d0 & 31) >> 2;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int k = kg * 4 + i;
                        blk[u][i] = make_float4(0.f, 0.f, 0.f, 0.f);
                        if (item < n_items && d0 < p.v_chunks * 32)
                            blk[u][i] = *reinterpret_cast<const float4 *>(src + ch * BN * 128 + k * 128 +
                                                                          ((unit ^ (k & 7)) << 4));
                    }
                }
#pragma unroll
                for (int u = 0; u < kMaxVItems; ++u) {
                    const int item = lt + u * kLoaderThreads;
                    if (item >= n_items) break;
                    const int kg = item % (BN / 4);
                    const int d0 = (item / (BN / 4)) * 4;
                    uint8_t *chunk = dst + (kg >> 3) * p.n_pv * 128;  // 32 keys per 128-byte V^T row chunk
                    const uint32_t unit = static_cast<uint32_t>(kg & 7);
                    const float4 c0 = make_float4(blk[u][0].x, blk[u][1].x, blk[u][2].x, blk[u][3].x);
                    const float4 c1 = make_float4(blk[u][0].y, blk[u][1].y, blk[u][2].y, blk[u][3].y);
                    const float4 c2 = make_float4(blk[u][0].z, blk[u][1].z, blk[u][2].z, blk[u][3].z);
                    const float4 c3 = make_float4(blk[u][0].w, blk[u][1].w, blk[u][2].w, blk[u][3].w);
                    *reinterpret_cast<float4 *>(chunk + (d0 + 0) * 128 + ((unit ^ ((d0 + 0) & 7)) << 4)) = c0;
                    *reinterpret_cast<float4 *>(chunk + (d0 + 1) * 128 + ((unit ^ ((d0 + 1) & 7)) << 4)) = c1;
                    *reinterpret_cast<float4 *>(chunk + (d0 + 2) * 128 + ((unit ^ ((d0 + 2) & 7)) << 4)) = c2;
                    *reinterpret_cast<float4 *>(chunk + (d0 + 3) * 128 + ((unit ^ ((d0 + 3) & 7)) << 4)) = c3;
                }
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                mbar_arrive(smem_u32(&ctl.full_v[st]));
            }
        }
    } else if (t < T && n_my > 0 && unit_ok) {
        // ------------------------------------------------------------ softmax warpgroup of tile t
        // Q_t into TMEM: this thread's row of the TMA-loaded tile (128-byte rows of 32 values per column chunk,
        // 16-byte units swizzled with the row), zero past D_qk and past S_q (TMA fills).
        {
            const bool qok = wait_bounded(smem_u32(&ctl.q_smem), 0, ctl.abort_flag, p);
            ok = __all_sync(0xffffffffu, qok);
            const uint32_t q_addr = tmem + lane_base + col_q0 + t * dq;
            const uint8_t *qsrc = smem_raw + (sQ - raw) + t * q_tile_bytes + row * 128;
            if (ok) {
                for (int c = 0; c < dq; c += 8) {
                    const uint8_t *chunk = qsrc + (c >> 5) * (kBM * 128);
                    const int u0 = (c & 31) >> 2;
                    const float4 a = *reinterpret_cast<const float4 *>(chunk + ((u0 ^ (row & 7)) << 4));
                    const float4 b = *reinterpret_cast<const float4 *>(chunk + (((u0 + 1) ^ (row & 7)) << 4));
                    const uint32_t w[8] = {__float_as_uint(a.x), __float_as_uint(a.y), __float_as_uint(a.z),
                                           __float_as_uint(a.w), __float_as_uint(b.x), __float_as_uint(b.y),
                                           __float_as_uint(b.z), __float_as_uint(b.w)};
                    tmem_st8(q_addr + c, w);
                }
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(smem_u32(&ctl.q_full[t]));
        }
        const uint32_t s_addr = tmem + lane_base + col_s0 + t * BN;
        const uint32_t o_addr = tmem + lane_base + col_o0 + t * p.n_pv;
        // Non-positive scales are applied to the scores first (FOLD false), so the folded form below sees c > 0.
        const float c = FOLD ? p.scale_log2 : 1.0f;
        const float2 c2 = make_float2(c, c);
        const int key_lo = band_key_lo(p, q_row), key_hi = band_key_hi(p, q_row);
        const int tile_row0 = U.r0 + t * kBM;
        const int mask_lo = band_key_lo(p, min(tile_row0 + kBM, p.S_q) - 1);
        const int mask_hi = band_key_hi(p, tile_row0);
        uint32_t s_par = 0;
        for (int j = 0; j < n_my; ++j) {
            ok = wait_bounded(smem_u32(&ctl.s_full[t]), s_par, ctl.abort_flag, p);
            s_par ^= 1u;
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
            uint32_t sr[BN];
            tmem_ld32(s_addr, sr);
            tmem_ld32(s_addr + 32, sr + 32);
            tmem_wait_ld();
            float x[BN];
#pragma unroll
            for (int k = 0; k < BN; ++k) x[k] = __uint_as_float(sr[k]);
            if constexpr (!FOLD) {
#pragma unroll
                for (int k = 0; k < BN; ++k) x[k] *= p.scale_log2;
            }
            const int k0 = (U.j0 + U.as[t] + j) * BN;
            if (k0 < mask_lo || k0 + BN > mask_hi) {
#pragma unroll
                for (int k = 0; k < BN; ++k)
                    if (k0 + k < key_lo || k0 + k >= key_hi) x[k] = -INFINITY;
            }
            float mx0 = fmax3(x[0], x[1], x[2]), mx1 = fmax3(x[3], x[4], x[5]);
            float mx2 = fmax3(x[6], x[7], x[8]), mx3 = fmax3(x[9], x[10], x[11]);
#pragma unroll
            for (int k = 12; k < BN - 4; k += 8) {
                mx0 = fmax3(mx0, x[k], x[k + 1]);
                mx1 = fmax3(mx1, x[k + 2], x[k + 3]);
                mx2 = fmax3(mx2, x[k + 4], x[k + 5]);
                mx3 = fmax3(mx3, x[k + 6], x[k + 7]);
            }
            mx0 = fmax3(mx0, x[BN - 4], x[BN - 3]);
            mx1 = fmax3(mx1, x[BN - 2], x[BN - 1]);
            const float m_tile = fmax3(fmaxf(mx0, mx1), mx2, mx3) * c;  // c > 0: -inf stays -inf
            const float m_new = fmaxf(m_used, m_tile);
            // lazy rescale: keep the old reference unless the max grew by more than tau
            const bool resc = (m_used == -INFINITY) ? (m_new != -INFINITY) : (m_new - m_used > kTau);
            float alpha = 1.0f;
            if (resc) {
                alpha = (m_used == -INFINITY) ? 0.0f : ex2(m_used - m_new);
                l *= alpha;
                m_used = m_new;
            }
            const float m_ref = (m_used == -INFINITY) ? 0.0f : m_used;
            const float2 nm2 = make_float2(-m_ref, -m_ref);
            // p = 2^(s * c - m_ref), the scale folded into one paired FMA per two scores
            float2 acc0 = make_float2(0.f, 0.f), acc1 = acc0;
            uint32_t pk[BN];
#pragma unroll
            for (int k = 0; k < BN; k += 4) {
                const float2 y0 = __ffma2_rn(make_float2(x[k], x[k + 1]), c2, nm2);
                const float2 y1 = __ffma2_rn(make_float2(x[k + 2], x[k + 3]), c2, nm2);
                const float2 e0 = make_float2(ex2(y0.x), ex2(y0.y));
                const float2 e1 = make_float2(ex2(y1.x), ex2(y1.y));
                acc0 = __fadd2_rn(acc0, e0);
                acc1 = __fadd2_rn(acc1, e1);
                pk[k] = __float_as_uint(e0.x);
                pk[k + 1] = __float_as_uint(e0.y);
                pk[k + 2] = __float_as_uint(e1.x);
                pk[k + 3] = __float_as_uint(e1.y);
            }
            l += (acc0.x + acc0.y) + (acc1.x + acc1.y);
            tmem_st32(s_addr, pk);  // P_t,j over S_t,j (fp32)
            tmem_st32(s_addr + 32, pk + 32);
            // O_t *= alpha where the reference moved.  The scores just read were committed after P_t,j-1 V_j-1,
            // so O_t holds its final value for tile j-1 and no MMA touches it now.
            if (j > 0 && __any_sync(0xffffffffu, resc)) {
                for (int cc = 0; cc < p.n_pv; cc += 16) {
                    uint32_t o[16];
                    tmem_ld16(o_addr + cc, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int k = 0; k < 16; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
                    tmem_st16(o_addr + cc, o);
                }
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(smem_u32(&ctl.p_full[t]));
        }
        if (ok) {
            ok = wait_bounded(smem_u32(&ctl.o_done[t]), 0, ctl.abort_flag, p);
            ok = __all_sync(0xffffffffu, ok);
        }
        if (ok) tc_fence_after();
    }
    __syncwarp();

    // ---------------------------------------------------------------- epilogue
    // A softmax thread's row holds O_t (unnormalised, in TMEM), m_used and l for this CTA's share of the
    // keys; `has` says whether the share gave the row any key tile (otherwise the partial is empty: O = 0,
    // m = -inf, l = 0, and TMEM holds nothing for it).  A CTA that stopped early (time-out, failed check)
    // writes nothing.  TMEM loads are warp-collective, so every condition around them is warp-uniform
    // (`row_active`, `live`, `has`; the cluster owner of a row is the same for the 32 rows of a warp), and
    // only the stores depend on the lane's row.
    const bool row_active = is_softmax && t < T;
    const bool live = unit_ok && __shfl_sync(0xffffffffu, ctl.abort_flag, 0) == 0;
    const bool has = row_active && n_my > 0 && ok && live;
    const bool row_ok = row_active && q_row < p.S_q;
    const uint32_t o_addr = tmem + lane_base + col_o0 + t * p.n_pv;

    // 16 columns of O_t from TMEM (zeros when the share gave the row no key tile).
    auto load_o = [&](int cc, float (&v)[16]) {
        uint32_t o[16];
        if (has) {
            tmem_ld16(o_addr + cc, o);
            tmem_wait_ld();
        }
#pragma unroll
        for (int k = 0; k < 16; ++k) v[k] = has ? __uint_as_float(o[k]) : 0.0f;
    };
    // Columns cc .. cc + 15 (those below D_v) of a row, times `scale`, with 16-byte stores where whole.
    auto store16 = [&](float *row_ptr, int cc, const float (&v)[16], float scale) {
#pragma unroll
        for (int k = 0; k < 16; k += 4) {
            const int d = cc + k;
            const float4 x = make_float4(v[k] * scale, v[k + 1] * scale, v[k + 2] * scale, v[k + 3] * scale);
            if (d + 4 <= p.D_v) {
                *reinterpret_cast<float4 *>(row_ptr + d) = x;
            } else if (d < p.D_v) {
                row_ptr[d] = x.x;
                if (d + 1 < p.D_v) row_ptr[d + 1] = x.y;
                if (d + 2 < p.D_v) row_ptr[d + 2] = x.z;
            }
        }
    };
    float *const orow = static_cast<float *>(p.O) + static_cast<long long>(U.b) * p.o_sb +
                        static_cast<long long>(U.h) * p.o_sh + static_cast<long long>(q_row) * p.o_ss;
    const long long lse_idx = (static_cast<long long>(U.b) * p.H + U.h) * p.S_q + q_row;

    if (p.cluster > 1) {
        // ------------------------------------------------------------ merge inside the cluster
        // CTA r of the cluster owns rows [r * R / C, (r + 1) * R / C) of the unit's R rows (R / C >= 32, whole
        // warps).  Once both softmax warpgroups are past their last P V (the ring is idle), every row's partial
        // (O, m, l) goes to a staging area in this CTA's ring memory; after a cluster barrier (every CTA's
        // ring is idle, so receiving is safe) one thread sends each other CTA the block of its rows with one
        // bulk copy, which completes on that CTA's recv_full barrier.  Each owner then combines the C partials
        // of its rows:  O = sum_c 2^(m_c - M) O_c / sum_c 2^(m_c - M) l_c,  M = max_c m_c.  A last cluster
        // barrier keeps every CTA's shared memory alive until all copies have landed.
        const int C = p.cluster;
        const int rank = static_cast<int>(cluster_ctarank());
        const int R = T * kBM;
        const int rows_per_owner = R / C;
        const int u = t * kBM + row;
        const int owner = u / rows_per_owner;
        const int n_out4 = (p.D_v + 3) / 4;
        const uint32_t rs = static_cast<uint32_t>(n_out4 + 1) * 16;  // a row: O (n_out4 float4), then m, l, 0, 0
        const uint32_t stage_area = base;                           // R rows, in unit order
        const uint32_t recv_area = base + R * rs;                   // C slots of rows_per_owner rows (own slot unused)
        uint8_t *const smem_gen = smem_raw + (base - raw);
        if (is_softmax) {
            named_bar_sync(1, 256);  // both tiles' products are done: the ring is idle
            if (row_active) {
                float4 *dst = reinterpret_cast<float4 *>(smem_gen + u * rs);
                for (int cc = 0; cc < p.D_v; cc += 16) {
                    float v[16];
                    load_o(cc, v);
#pragma unroll
                    for (int k = 0; k < 16; k += 4)
                        if (cc + k < p.D_v) dst[(cc + k) / 4] = make_float4(v[k], v[k + 1], v[k + 2], v[k + 3]);
                }
                dst[n_out4] = make_float4((has && l > 0.0f) ? m_used : -INFINITY, has ? l : 0.0f, 0.0f, 0.0f);
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // the staged rows feed bulk copies
            named_bar_sync(1, 256);
            if (warp == 4 && lane == 0)
                mbar_arrive_expect_tx(smem_u32(&ctl.recv_full), static_cast<uint32_t>((C - 1) * rows_per_owner) * rs);
        }
        cluster_sync();
        if (warp == 4 && lane == 0) {
            for (int o = 0; o < C; ++o) {
                if (o == rank) continue;
                bulk_copy_to_cluster(cluster_map(recv_area + static_cast<uint32_t>(rank * rows_per_owner) * rs, o),
                                     stage_area + static_cast<uint32_t>(o * rows_per_owner) * rs,
                                     static_cast<uint32_t>(rows_per_owner) * rs,
                                     cluster_map(smem_u32(&ctl.recv_full), o));
            }
        }
        if (row_active && owner == rank && live) {
            const bool got = __all_sync(0xffffffffu, wait_bounded(smem_u32(&ctl.recv_full), 0, ctl.abort_flag, p));
            const int u_local = u - rank * rows_per_owner;
            auto rec = [&](int src) {  // partial row of source CTA src (this CTA's own from its staging area)
                return reinterpret_cast<const float4 *>(
                    smem_gen + (src == rank ? static_cast<uint32_t>(u) * rs
                                            : R * rs + static_cast<uint32_t>(src * rows_per_owner + u_local) * rs));
            };
            float ms[kMaxCluster], ls[kMaxCluster];
            float M = -INFINITY;
#pragma unroll
            for (int src = 0; src < kMaxCluster; ++src) {
                const float4 ml = src < C ? rec(src)[n_out4] : make_float4(-INFINITY, 0.f, 0.f, 0.f);
                ms[src] = ml.x;
                ls[src] = ml.y;
                M = fmaxf(M, ml.x);
            }
            float L = 0.0f, w[kMaxCluster];
#pragma unroll
            for (int src = 0; src < kMaxCluster; ++src) {
                w[src] = ms[src] != -INFINITY ? ex2(ms[src] - M) : 0.0f;  // a share without keys weighs 0 (its O is 0)
                L += w[src] * ls[src];
            }
            const float inv = L > 0.0f ? 1.0f / L : 0.0f;  // no share saw a key of this row: it is 0
#pragma unroll
            for (int src = 0; src < kMaxCluster; ++src) w[src] *= inv;
            if (got && row_ok) {
                for (int g = 0; g < n_out4; ++g) {
                    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                    for (int src = 0; src < kMaxCluster; ++src) {
                        if (src < C) {
                            const float4 x = rec(src)[g];
                            acc.x += w[src] * x.x;
                            acc.y += w[src] * x.y;
                            acc.z += w[src] * x.z;
                            acc.w += w[src] * x.w;
                        }
                    }
                    const int d = g * 4;
                    if (d + 4 <= p.D_v) {
                        *reinterpret_cast<float4 *>(orow + d) = acc;
                    } else {
                        orow[d] = acc.x;
                        if (d + 1 < p.D_v) orow[d + 1] = acc.y;
                        if (d + 2 < p.D_v) orow[d + 2] = acc.z;
                    }
                }
                if (p.lse) p.lse[lse_idx] = lse_from(M, L);
            }
        }
        __syncwarp();
        cluster_sync();
    } else if (p.n_split > 1) {
        // ------------------------------------------------------------ partial result for the merge kernel
        if (row_active && live) {
            const long long part = static_cast<long long>(U.share) * p.B * p.H * p.S_q + lse_idx;
            float *prow = p.part_o + part * p.D_v;
            for (int cc = 0; cc < p.D_v; cc += 16) {
                float v[16];
                load_o(cc, v);
                if (row_ok) store16(prow, cc, v, 1.0f);
            }
            if (row_ok) {
                p.part_m[part] = has ? m_used : -INFINITY;
                p.part_l[part] = has ? l : 0.0f;
                p.part_c[part] = 0.0f;  // P stays fp32 here: no bf16 rounding to weigh
            }
        }
    } else if (row_active && live) {
        // ------------------------------------------------------------ O = O_t / l
        const float inv = (has && l > 0.0f) ? 1.0f / l : 0.0f;  // a row without keys is written as 0
        for (int cc = 0; cc < p.D_v; cc += 16) {
            float v[16];
            load_o(cc, v);
            if (row_ok) store16(orow, cc, v, inv);
        }
        if (p.lse && row_ok) p.lse[lse_idx] = lse_from(has ? m_used : -INFINITY, has ? l : 0.0f);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

}  // namespace vt
