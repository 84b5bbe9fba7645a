// Attention forward kernel for sm_103a: O = softmax(scale * Q K^T) V per (batch, head).
//
// One CTA computes one work item: a 128-row query block of one (b, h) slice.  Warp roles:
//   warp 0      TMA producer: the Q block once, then K and V tiles of BN keys through a
//               `stages`-deep ring of shared-memory slots (mbarrier full/empty pairs).
//   warp 1      TMEM owner and MMA issuer (the whole warp; one elected lane issues): S_j = Q K_j^T
//               into a TMEM score buffer (two buffers, alternating), then O += P_j V_j with P_j
//               read from TMEM.
//   warps 2-5   softmax warpgroup, one query row per thread: S_j from TMEM, masks, running
//               max with lazy rescaling, exp2 with the folded scale, P_j back into TMEM
//               over S_j, O rescale when the reference max moves, and the epilogue.
//   warps 6-15  fp32 I/O only: V loaders, two groups of four warps taking alternate key tiles
//               (warps 9 and 13 idle: no loader on the MMA warp's sub-partition).  The TF32 MMA takes its B operand K-major only (an
//               N-major tf32 B reads as zeros), so V tiles are read with coalesced 16-byte
//               loads and written transposed (keys contiguous) into the 128-byte-swizzled
//               K-major layout; for bf16, V goes by TMA as it is (N-major B).
//
// The tiling follows the FA-1 boundary kernel of the VeriTile page
// "VeriTile.Examples.FlashAttention1.NaiveRefinement" (M query rows per program, key
// blocks of Bk, a head tile of Bd >= D, writes only where row < S_q and d < D); the four
// reductions are the accy page's score_dot, score_max, score_exp_sum and
// value_weighted_sum, computed online; the exp2-with-folded-scale form is the "Base-2
// scaled attention" of the VeriTile coverage table (sm_scale * log2(e)).
#pragma once

#include <cuda.h>
#include <cstdint>

#include "vt_attn_common.cuh"

namespace vt {

template <int DT>
struct Cfg {
    static constexpr int kElt = DT == kBF16 ? 2 : 4;
    static constexpr int kBN = DT == kBF16 ? 128 : 64;         // keys per tile
    static constexpr int kKStep = DT == kBF16 ? 16 : 8;        // MMA K per instruction
    static constexpr int kChunkElems = 128 / kElt;             // elements per 128-byte chunk
    static constexpr uint32_t kFmt = DT == kBF16 ? 1u : 2u;    // bf16 / tf32
    static constexpr uint32_t kTmemCols = DT == kBF16 ? 512u : 256u;
    static constexpr uint32_t kColS0 = 0, kColS1 = kBN, kColO = 2 * kBN;
    // fp32: two V-loader groups of 128 threads take alternate key tiles, so two tiles' global
    // reads are in flight at once (one group alone was bound by one read round trip per tile).
    static constexpr int kVLoaderGroups = DT == kBF16 ? 0 : 2;
    static constexpr int kVLoaders = DT == kBF16 ? 0 : 128;  // threads per group
    // fp32: warps 6-15, of which 9 and 13 stay idle so that no loader shares sub-partition 1 with
    // the MMA warp (16 warps cost no more registers per thread than 14)
    static constexpr int kThreads = DT == kBF16 ? 192 : 512;
    // float4 loads per loader thread and V tile, at most (BN keys x 128 columns / 4 / loaders)
    static constexpr int kVLoadsPerThread = DT == kBF16 ? 1 : (64 * 128 / 4) / 128;
};

// Bytes of one V stage: bf16 keeps V N-major (128-byte column chunks of BN key rows); fp32
// stores V^T K-major (n_pv rows of BN keys, in 128-byte key chunks).
template <int DT>
__host__ __device__ inline int v_stage_bytes(int v_chunks, int n_pv) {
    return DT == kBF16 ? v_chunks * Cfg<DT>::kBN * 128 : n_pv * Cfg<DT>::kBN * 4;
}

// Byte offset of (row r, byte c) in a 1024-byte-aligned region of 128-byte rows laid out
// the way the 128-byte TMA swizzle lays them out: 16-byte unit index XOR (row mod 8).
__device__ __forceinline__ uint32_t swizzle128(int r, int c) {
    return static_cast<uint32_t>(r * 128 + ((((c >> 4) ^ (r & 7))) << 4) + (c & 15));
}

struct SharedCtl {
    uint64_t full_k[kMaxStages];
    uint64_t full_v[kMaxStages];
    uint64_t empty[kMaxStages];
    uint64_t q_full;
    uint64_t s_full[2];
    uint64_t p_full[2];
    uint64_t o_done[2];  // P_j V_j done, for j even / odd
    uint64_t drain;
    uint64_t stall;
    uint32_t tmem_base;
    volatile uint32_t abort_flag;
};

// KQ: MMA K-steps (8 tf32 each) of Q K^T, D_qk rounded up to a whole 128-byte chunk: 4, 8, 12 or 16.
template <int DT, int KQ>
__global__ void __launch_bounds__(Cfg<DT>::kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const AttnParams p) {
    using C = Cfg<DT>;
    constexpr int BN = C::kBN;
    __shared__ SharedCtl ctl;
    extern __shared__ uint8_t smem_raw[];

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // Work item: all heads' heaviest query blocks first when work grows with the block index;
    // with split-KV, the n_split shares of one item are adjacent in the launch order.
    const int split = blockIdx.x % p.n_split;
    const int item = blockIdx.x / p.n_split;
    const int bh_count = p.B * p.H;
    const int slot = item / bh_count;
    const int bh = item - slot * bh_count;
    const int qb = p.reverse_q ? (p.n_qblocks - 1 - slot) : slot;
    const int h = bh % p.H;
    const int b = bh / p.H;
    const int hk = h / p.kv_group;  // key/value head
    const int q_row0 = qb * kBM;
    // key tiles [j_first, j_first + n_kv) that some row of the block may see (none: n_kv = 0)
    // and this CTA's contiguous share of them
    int j_first, j_end;
    band_tiles(p, q_row0, min(q_row0 + kBM, p.S_q) - 1, BN, &j_first, &j_end);
    const int n_all = j_end - j_first;
    const int per = (n_all + p.n_split - 1) / p.n_split;
    const int share_lo = min(split * per, n_all);
    j_first += share_lo;
    const int n_kv = min(n_all, share_lo + per) - share_lo;
    // (checked by the debug build before any load of the item)
    auto item_valid = [&]() {
        return split >= 0 && split < p.n_split && qb >= 0 && qb < p.n_qblocks && b >= 0 && b < p.B && h >= 0 &&
               h < p.H && hk == h / p.kv_group && q_row0 < p.S_q && j_first >= 0 && n_kv >= 0 &&
               j_first + n_kv <= (p.S_k + BN - 1) / BN;
    };

    // Shared-memory carve-up (1024-byte aligned for the 128-byte swizzle).
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const uint32_t q_bytes = p.q_chunks * kBM * 128;
    const uint32_t k_bytes = p.q_chunks * BN * 128;
    const uint32_t v_bytes = v_stage_bytes<DT>(p.v_chunks, p.n_pv);
    const uint32_t sQ = base;
    auto sK = [&](int st) { return base + q_bytes + st * (k_bytes + v_bytes); };
    auto sV = [&](int st) { return base + q_bytes + st * (k_bytes + v_bytes) + k_bytes; };

    if (threadIdx.x == 0) {
        for (int s = 0; s < p.stages; ++s) {
            mbar_init(smem_u32(&ctl.full_k[s]), 1);
            mbar_init(smem_u32(&ctl.full_v[s]), DT == kBF16 ? 1 : C::kVLoaders);
            mbar_init(smem_u32(&ctl.empty[s]), 1);
        }
        mbar_init(smem_u32(&ctl.q_full), 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&ctl.s_full[i]), 1);
            mbar_init(smem_u32(&ctl.p_full[i]), 128);
        }
        mbar_init(smem_u32(&ctl.o_done[0]), 1);
        mbar_init(smem_u32(&ctl.o_done[1]), 1);
        mbar_init(smem_u32(&ctl.drain), 1);
        mbar_init(smem_u32(&ctl.stall), 1);
        ctl.abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&ctl.tmem_base), C::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctl.tmem_base;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0 && n_kv > 0 &&
            VT_DEV_CHECK(!(p.flags & kFlagTestBounds) && item_valid(), ctl.abort_flag, p)) {  // else nothing issued
            mbar_arrive_expect_tx(smem_u32(&ctl.q_full), q_bytes);
            for (int c = 0; c < p.q_chunks; ++c)
                tma_load_4d(sQ + c * kBM * 128, &tmQ, smem_u32(&ctl.q_full), c * C::kChunkElems, q_row0, h, b);
            int issued = 0;
            for (int j = 0; j < n_kv; ++j) {
                const int st = j % p.stages;
                const int use = j / p.stages;
                if (use > 0 && !wait_bounded(smem_u32(&ctl.empty[st]), (use - 1) & 1, ctl.abort_flag, p)) break;
                mbar_arrive_expect_tx(smem_u32(&ctl.full_k[st]), k_bytes);
                for (int c = 0; c < p.q_chunks; ++c)
                    tma_load_4d(sK(st) + c * BN * 128, &tmK, smem_u32(&ctl.full_k[st]), c * C::kChunkElems,
                                (j_first + j) * BN, hk, b);
                if (DT == kBF16) {
                    mbar_arrive_expect_tx(smem_u32(&ctl.full_v[st]), v_bytes);
                    for (int c = 0; c < p.v_chunks; ++c)
                        tma_load_4d(sV(st) + c * BN * 128, &tmV, smem_u32(&ctl.full_v[st]), c * C::kChunkElems,
                                    (j_first + j) * BN, hk, b);
                }
                issued = j + 1;
            }
            if (ctl.abort_flag) {
                // Let every copy this thread started land before the CTA's memory goes away.
                wait_drain(smem_u32(&ctl.q_full), 0, p);
                for (int j = max(0, issued - p.stages); j < issued; ++j) {
                    const int st = j % p.stages;
                    wait_drain(smem_u32(&ctl.full_k[st]), (j / p.stages) & 1, p);
                    if (DT == kBF16) wait_drain(smem_u32(&ctl.full_v[st]), (j / p.stages) & 1, p);
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        // Descriptors are built once as (low, high) words and the K-steps are unrolled (KQ).  The
        // whole warp runs this code with warp-uniform values and waits on every barrier; one lane
        // chosen by elect.sync issues each MMA and commit.
        if (n_kv > 0) {
            static_assert(DT == kF32, "this kernel serves fp32 I/O; bf16 uses the two-tile kernel");
            const uint32_t idesc_qk = instr_desc(C::kFmt, kBM, BN, 0);
            const uint32_t idesc_pv = instr_desc(C::kFmt, kBM, p.n_pv, 0);
            const uint64_t qdesc = smem_desc_sw128(sQ, 16, 1024);
            const uint64_t kdesc0 = smem_desc_sw128(sK(0), 16, 1024);
            const uint64_t vdesc0 = smem_desc_sw128(sV(0), 16, 1024);  // V^T, K-major
            const uint32_t q_lo = static_cast<uint32_t>(qdesc), q_hi = static_cast<uint32_t>(qdesc >> 32);
            const uint32_t k_lo0 = static_cast<uint32_t>(kdesc0), k_hi = static_cast<uint32_t>(kdesc0 >> 32);
            const uint32_t v_lo0 = static_cast<uint32_t>(vdesc0), v_hi = static_cast<uint32_t>(vdesc0 >> 32);
            const uint32_t stage_step = (k_bytes + v_bytes) >> 4;
            const uint32_t v_chunk = static_cast<uint32_t>(p.n_pv) * 8;  // one V^T key chunk, descriptor units
            bool ok = true, any_mma = false;
            // Every lane waits, so whichever lane elect.sync picks has itself observed the phase.
            auto wait1 = [&](uint32_t bar, uint32_t parity) -> bool {
                return __all_sync(0xffffffffu, wait_bounded(bar, parity, ctl.abort_flag, p)) != 0;
            };
            if (p.flags & kFlagTestStall) ok = wait1(smem_u32(&ctl.stall), 0);  // test hook: never signalled
            if (ok) ok = wait1(smem_u32(&ctl.q_full), 0);

            auto issue_qk = [&](int j) -> bool {
                const int st = j % p.stages;
                if (!wait1(smem_u32(&ctl.full_k[st]), (j / p.stages) & 1)) return false;
                const uint32_t d = tmem + ((j & 1) ? C::kColS1 : C::kColS0);
                const uint32_t k_lo = k_lo0 + st * stage_step;
#pragma unroll
                for (int kk = 0; kk < KQ; ++kk)
                    mma_ss_tf32_elect(d, q_lo + (kk >> 2) * (kBM * 8) + (kk & 3) * 2, q_hi,
                                  k_lo + (kk >> 2) * (BN * 8) + (kk & 3) * 2, k_hi, idesc_qk, kk > 0);
                mma_commit_elect(smem_u32(&ctl.s_full[j & 1]));
                any_mma = true;
                return true;
            };

            if (ok) ok = issue_qk(0);
            for (int j = 0; ok && j < n_kv; ++j) {
                if (j + 1 < n_kv && !issue_qk(j + 1)) { ok = false; break; }
                const int st = j % p.stages;
                if (!wait1(smem_u32(&ctl.p_full[j & 1]), (j >> 1) & 1)) { ok = false; break; }
                if (!wait1(smem_u32(&ctl.full_v[st]), (j / p.stages) & 1)) { ok = false; break; }
                tc_fence_after();  // P was written to TMEM and V^T to shared memory by other warps
                const uint32_t a_base = tmem + ((j & 1) ? C::kColS1 : C::kColS0);
                const uint32_t v_lo = v_lo0 + st * stage_step;
                // V^T K-major: K-step = 8 keys = 32 bytes inside a 128-byte key chunk
#pragma unroll
                for (int kk = 0; kk < BN / C::kKStep; ++kk)
                    mma_ts_tf32_elect(tmem + C::kColO, a_base + kk * 8, v_lo + (kk >> 2) * v_chunk + (kk & 3) * 2, v_hi,
                                  idesc_pv, (j > 0 || kk > 0));
                mma_commit_elect(smem_u32(&ctl.empty[st]));
                mma_commit_elect(smem_u32(&ctl.o_done[j & 1]));
            }
            if (!ok && any_mma) {
                mma_commit_elect(smem_u32(&ctl.drain));
                if (lane == 0) wait_drain(smem_u32(&ctl.drain), 0, p);
                __syncwarp();
            }
        }
    } else if (DT == kF32 && warp >= 6) {
        // ------------------------------------------------------------ fp32 V loader (transposing)
      if (warp != 9 && warp != 13) {  // warps 9 and 13 stay idle
        const int wl = warp - 6;
        const int li = wl - (wl > 3) - (wl > 7);               // loader warp 0..7
        const int group = li >> 2;                             // takes key tiles j = group (mod groups)
        const int lt = (li & 3) * 32 + lane;
        const int nd4 = p.n_pv / 4;  // 4-column groups, including the zero padding up to n_pv
        const float *vbh = static_cast<const float *>(p.V) + static_cast<long long>(b) * p.v_sb +
                           static_cast<long long>(hk) * p.v_sh;
        uint8_t *smem_gen = smem_raw + (base - raw);
        const bool loads_ok = VT_DEV_CHECK(item_valid(), ctl.abort_flag, p);
        for (int j = group; loads_ok && j < n_kv; j += C::kVLoaderGroups) {
            const int st = j % p.stages;
            const int use = j / p.stages;
            if (use > 0) {
                bool ok = wait_bounded(smem_u32(&ctl.empty[st]), (use - 1) & 1, ctl.abort_flag, p);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
            }
            uint8_t *dst = smem_gen + (sV(st) - base);
            // All of this thread's loads of the tile are issued before any store, so the tile
            // costs one memory round trip rather than one per load.  An item is a block of 4 keys
            // x 4 columns: four 16-byte row loads, a register transpose, and four 16-byte stores
            // of 4 consecutive keys of one column (16 contiguous bytes of V^T, which the 128-byte
            // swizzle keeps together).  Items run key-group fastest, so each 8-lane store phase
            // covers 8 different 16-byte units of a row.
            constexpr int kItems = C::kVLoadsPerThread / 4;  // 4x4 blocks per thread, at most
            float4 blk[kItems][4];
            const int n_items = (BN / 4) * nd4;
#pragma unroll
            for (int u = 0; u < kItems; ++u) {
                const int item = lt + u * C::kVLoaders;
                const int kg = item % (BN / 4);
                const int d0 = (item / (BN / 4)) * 4;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int kglob = (j_first + j) * BN + kg * 4 + i;
                    blk[u][i] = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (item < n_items && kglob < p.S_k && d0 < p.D_v) {
                        const float *src = vbh + static_cast<long long>(kglob) * p.v_ss + d0;
                        if (d0 + 4 <= p.D_v) {
                            blk[u][i] = __ldg(reinterpret_cast<const float4 *>(src));
                        } else {
                            blk[u][i].x = __ldg(src);
                            if (d0 + 1 < p.D_v) blk[u][i].y = __ldg(src + 1);
                            if (d0 + 2 < p.D_v) blk[u][i].z = __ldg(src + 2);
                        }
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < kItems; ++u) {
                const int item = lt + u * C::kVLoaders;
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
    } else {
        // ------------------------------------------------------------ softmax warpgroup
        const int quad = warp & 3;                 // TMEM lane quadrant this warp may access
        const int row = quad * 32 + lane;          // row of the query block owned by this thread
        const int q_row = q_row0 + row;
        const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
        const float c = p.scale_log2;
        // this row's allowed keys [key_lo, key_hi); a key tile starting below mask_lo or ending past
        // mask_hi cuts some row's range and is masked (the same decision for the whole warpgroup)
        const int key_lo = band_key_lo(p, q_row), key_hi = band_key_hi(p, q_row);
        const int mask_lo = band_key_lo(p, min(q_row0 + kBM, p.S_q) - 1);
        const int mask_hi = band_key_hi(p, q_row0);
        float m_used = -INFINITY;  // reference max (log2 units) of O and l
        float l = 0.0f;
        bool ok = true;

        for (int j = 0; j < n_kv; ++j) {
            ok = wait_bounded(smem_u32(&ctl.s_full[j & 1]), (j >> 1) & 1, ctl.abort_flag, p);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
            const uint32_t s_addr = tmem + lane_base + ((j & 1) ? C::kColS1 : C::kColS0);
            uint32_t sr[BN];
#pragma unroll
            for (int cc = 0; cc < BN / 32; ++cc) tmem_ld32(s_addr + cc * 32, sr + cc * 32);
            tmem_wait_ld();

            float x[BN];
#pragma unroll
            for (int k = 0; k < BN; ++k) x[k] = __uint_as_float(sr[k]) * c;
            const int k0 = (j_first + j) * BN;
            if (k0 < mask_lo || k0 + BN > mask_hi) {
#pragma unroll
                for (int k = 0; k < BN; ++k)
                    if (k0 + k < key_lo || k0 + k >= key_hi) x[k] = -INFINITY;
            }
            float mx0 = x[0], mx1 = x[1], mx2 = x[2], mx3 = x[3];
#pragma unroll
            for (int k = 4; k < BN; k += 4) {
                mx0 = fmaxf(mx0, x[k]);
                mx1 = fmaxf(mx1, x[k + 1]);
                mx2 = fmaxf(mx2, x[k + 2]);
                mx3 = fmaxf(mx3, x[k + 3]);
            }
            const float m_tile = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3));
            const float m_new = fmaxf(m_used, m_tile);
            // Lazy rescale: keep the old reference unless the max grew by more than tau.
            const bool resc = (m_used == -INFINITY) ? (m_new != -INFINITY) : (m_new - m_used > kRescaleTau);
            float alpha = 1.0f;
            if (resc) {
                alpha = (m_used == -INFINITY) ? 0.0f : ex2(m_used - m_new);
                l *= alpha;
                m_used = m_new;
            }
            const float m_ref = (m_used == -INFINITY) ? 0.0f : m_used;
            float l0 = 0.f, l1 = 0.f, l2 = 0.f, l3 = 0.f;
#pragma unroll
            for (int k = 0; k < BN; k += 4) {
                x[k] = ex2(x[k] - m_ref);
                x[k + 1] = ex2(x[k + 1] - m_ref);
                x[k + 2] = ex2(x[k + 2] - m_ref);
                x[k + 3] = ex2(x[k + 3] - m_ref);
                l0 += x[k];
                l1 += x[k + 1];
                l2 += x[k + 2];
                l3 += x[k + 3];
            }
            l += (l0 + l1) + (l2 + l3);

            // P_j over S_j in TMEM: bf16 pairs packed two per column, or fp32 one per column.
            if (DT == kBF16) {
                uint32_t pk[BN / 2];
#pragma unroll
                for (int k = 0; k < BN / 2; ++k) pk[k] = pack_bf16x2(x[2 * k], x[2 * k + 1]);
#pragma unroll
                for (int cc = 0; cc < BN / 64; ++cc) tmem_st32(s_addr + cc * 32, pk + cc * 32);
            } else {
                uint32_t pk[BN];
#pragma unroll
                for (int k = 0; k < BN; ++k) pk[k] = __float_as_uint(x[k]);
#pragma unroll
                for (int cc = 0; cc < BN / 32; ++cc) tmem_st32(s_addr + cc * 32, pk + cc * 32);
            }

            // O *= alpha for rows whose reference moved, once P_{j-1} V_{j-1} has landed.  That
            // wait sits before the hand-over of P_j only when a row rescales; otherwise the phase
            // is consumed after the hand-over, off the chain S_j -> P_j -> P_j V_j.  With one
            // barrier per parity of j, o_done[(j-1) & 1] cannot complete again before P_{j+1} is
            // handed over, so a late wait never sees an ambiguous phase.
            const bool fix_o = j > 0 && __any_sync(0xffffffffu, resc);
            if (fix_o) {
                ok = wait_bounded(smem_u32(&ctl.o_done[(j - 1) & 1]), ((j - 1) >> 1) & 1, ctl.abort_flag, p);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                tc_fence_after();
                const uint32_t o_addr = tmem + lane_base + C::kColO;
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
            mbar_arrive(smem_u32(&ctl.p_full[j & 1]));
            if (j > 0 && !fix_o) {
                ok = wait_bounded(smem_u32(&ctl.o_done[(j - 1) & 1]), ((j - 1) >> 1) & 1, ctl.abort_flag, p);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
            }
        }

        if (ok && n_kv > 0) {
            ok = wait_bounded(smem_u32(&ctl.o_done[(n_kv - 1) & 1]), ((n_kv - 1) >> 1) & 1, ctl.abort_flag, p);
            ok = __all_sync(0xffffffffu, ok);
        }
        if (ok) {
            // ------------------------------------------------------------ epilogue
            // A row with no allowed key (l = 0, or no key tile at all) is written as 0; with
            // split-KV the share writes its unnormalised O with its reference max m (log2 units)
            // and sum l instead (the empty share: O = 0, m = -inf, l = 0), and the merge kernel
            // finishes the row.
            if (n_kv > 0) tc_fence_after();
            if (p.n_split > 1) {
                const uint32_t o_addr = tmem + lane_base + C::kColO;
                const bool row_ok = q_row < p.S_q;
                const long long row_lin = (static_cast<long long>(b) * p.H + h) * p.S_q + q_row;
                const long long part = static_cast<long long>(split) * p.B * p.H * p.S_q + row_lin;
                float *prow = p.part_o + part * p.D_v;
                for (int cc = 0; cc < p.n_pv; cc += 16) {
                    uint32_t o[16];
                    if (n_kv > 0) {
                        tmem_ld16(o_addr + cc, o);
                        tmem_wait_ld();
                    } else {
#pragma unroll
                        for (int k = 0; k < 16; ++k) o[k] = 0u;
                    }
                    if (!row_ok) continue;
                    if (cc + 16 <= p.D_v) {
                        float4 *dst = reinterpret_cast<float4 *>(prow + cc);
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            dst[k] = make_float4(__uint_as_float(o[4 * k]), __uint_as_float(o[4 * k + 1]),
                                                 __uint_as_float(o[4 * k + 2]), __uint_as_float(o[4 * k + 3]));
                    } else {
#pragma unroll
                        for (int k = 0; k < 16; ++k)
                            if (cc + k < p.D_v) prow[cc + k] = __uint_as_float(o[k]);
                    }
                }
                if (row_ok) {
                    p.part_m[part] = n_kv > 0 ? m_used : -INFINITY;
                    p.part_l[part] = n_kv > 0 ? l : 0.0f;
                    p.part_c[part] = 0.0f;  // P stays fp32 here: no bf16 rounding to weigh
                }
            } else {
            const float inv_l = l > 0.0f ? 1.0f / l : 0.0f;
            const uint32_t o_addr = tmem + lane_base + C::kColO;
            const bool row_ok = q_row < p.S_q;
            uint8_t *orow = reinterpret_cast<uint8_t *>(p.O) +
                            (static_cast<long long>(b) * p.o_sb + static_cast<long long>(h) * p.o_sh +
                             static_cast<long long>(q_row) * p.o_ss) * C::kElt;
            for (int cc = 0; cc < p.n_pv; cc += 16) {
                uint32_t o[16];
                if (n_kv > 0) {
                    tmem_ld16(o_addr + cc, o);
                    tmem_wait_ld();
                } else {
#pragma unroll
                    for (int k = 0; k < 16; ++k) o[k] = 0u;
                }
                if (!row_ok) continue;
                float v[16];
#pragma unroll
                for (int k = 0; k < 16; ++k) v[k] = __uint_as_float(o[k]) * inv_l;
                if (DT == kBF16) {
                    uint32_t w[8];
#pragma unroll
                    for (int k = 0; k < 8; ++k) w[k] = pack_bf16x2(v[2 * k], v[2 * k + 1]);
                    if (cc + 16 <= p.D_v) {
                        uint4 *dst = reinterpret_cast<uint4 *>(orow + cc * 2);
                        dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
                        dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
                    } else {
                        uint16_t *dst = reinterpret_cast<uint16_t *>(orow) + cc;
#pragma unroll
                        for (int k = 0; k < 16; ++k)
                            if (cc + k < p.D_v) dst[k] = static_cast<uint16_t>((w[k >> 1] >> ((k & 1) * 16)) & 0xFFFFu);
                    }
                } else {
                    if (cc + 16 <= p.D_v) {
                        float4 *dst = reinterpret_cast<float4 *>(orow + cc * 4);
#pragma unroll
                        for (int k = 0; k < 4; ++k) dst[k] = make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
                    } else {
                        float *dst = reinterpret_cast<float *>(orow) + cc;
#pragma unroll
                        for (int k = 0; k < 16; ++k)
                            if (cc + k < p.D_v) dst[k] = v[k];
                    }
                }
            }
            if (p.lse && row_ok)
                p.lse[(static_cast<long long>(b) * p.H + h) * p.S_q + q_row] = lse_from(m_used, l);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, C::kTmemCols);
    }
}

}  // namespace vt
