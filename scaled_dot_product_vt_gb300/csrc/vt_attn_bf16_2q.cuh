// Attention forward, bf16 I/O, for sm_103a: two 128-row query tiles per work unit sharing every
// 128-key K/V tile, one softmax warpgroup per query tile, tcgen05 issued by one warp (two warps, one
// per query tile, for value widths up to 64), one lane (elected once) issuing every MMA and commit.
//
// Persistent through cluster launch control: the grid has one CTA per work unit, but a running CTA
// takes over the units of CTAs that have not started yet (clusterlaunchcontrol.try_cancel), so about
// one CTA per SM runs and each one works through units in launch order (the producer warp obtains
// them and passes them to the other roles through a small ring in shared memory); the heavy units that
// come first spread over the SMs as they free up.  No state is shared between launches.
// A unit is 256 query rows of one (b, h) slice, as query tiles t = 0, 1 (rows r0 + 128 t ..
// r0 + 128 t + 127), and one share of their key tiles.  TMEM, barriers and descriptors live
// for the whole CTA; every barrier's phase is counted across units, so the producer loads the
// next unit's Q and K/V while the current unit's last tiles and epilogue run.
// Warp roles (12 warps, three warpgroups):
//   warp 0       TMA producer: per unit the Q tiles that have work (once the previous unit's last
//                Q K^T has read Q), then K_0, V_0, K_1, V_1, ... through a ring of equal
//                shared-memory slots (mbarrier full/empty per slot) that runs on across units.
//   warp 1       TMEM owner and MMA issuer (the whole warp runs the issuing code with warp-uniform
//                values; one lane, elected once, issues).  Per key tile j the tensor core runs
//                  O_0 += P_0,j V_j,  S_0 = Q_0 K_{j+1}^T,  O_1 += P_1,j V_j,  S_1 = Q_1 K_{j+1}^T
//                so while softmax warpgroup t works on S_t, the tensor core works for the other
//                tile.  Every operand descriptor is computed once; the K-steps are unrolled
//                (a per-instruction descriptor computation made the issuing thread, not the
//                tensor core, the bottleneck).
//                For value widths up to 64 (the score-ring variant) warp 1 issues for tile 0 and
//                warp 2 for tile 1, each one key tile ahead: S_t = Q_t K_{j+1}^T goes into a free
//                slot of tile t's ring while softmax t still works on S_t,j.
//   warps 2-3    idle (they complete warpgroup 0, which gives registers to the softmax warpgroups);
//                warp 2 is tile 1's issuer in the score-ring variant
//   warps 4-7    softmax warpgroup of tile 0, one row per thread (TMEM lane quadrant = warp % 4)
//   warps 8-11   softmax warpgroup of tile 1
// Registers: launched at 168 per thread; warpgroup 0 shrinks to 72 and the softmax warpgroups
// grow to 216 (128 x 72 + 256 x 216 = 384 x 168, so the increase never waits on a shortfall).
// TMEM (512 columns): S_0, S_1, O_0, O_1, 128 columns each (score ring: three 64-column score
// slots per tile at columns 0-191 and 192-383, O_0 and O_1 at 384 and 448; even key tiles put S in
// slots 0-1 and P in slot 0, odd ones S in slots 1-2 and P in slot 2, so the next scores never land
// on a P still being read).  P_t,j overwrites S_t,j as bf16
// pairs (64 columns) and is read from TMEM by the P V product.  Without the ring, a commit after S_t = Q_t K^T
// also covers the P V issued before it, so when softmax t sees its next scores, O_t is final
// for the previous tile and may be rescaled in place.  Softmax t reads O_t for a unit's epilogue
// before it hands over the next unit's first P_t, and the first P_t V of a unit (which overwrites
// O_t) waits for that hand-over: no separate barrier guards O_t between units.  With the ring the
// scores run a key tile ahead of P V, so each P V instead commits its own barrier (o_ready), and the
// softmax waits on it before rescaling O_t or reading it for the epilogue.
//
// The decomposition (query block, head, batch), the tail masks and the write set follow the
// FA-1 boundary kernel verified on the VeriTile page "VeriTile.Examples.FlashAttention1.
// NaiveRefinement"; the reductions are the accy page's score_dot, score_max, score_exp_sum and
// value_weighted_sum, computed online with the base-2 exponential of the folded scale.
#pragma once

#include "vt_attn_common.cuh"

namespace vt {
namespace q2 {

constexpr int kBN = 128;            // keys per tile
constexpr int kRows = 256;          // query rows per CTA
constexpr int kThreads = 384;       // 12 warps
constexpr int kRegsControl = 72;    // warpgroup 0 after setmaxnreg
constexpr int kRegsSoftmax = 216;   // softmax warpgroups after setmaxnreg
static_assert(128 * kRegsControl + 256 * kRegsSoftmax <= kThreads * 168, "register split exceeds the launch");
constexpr int kMaxSlots = 6;
constexpr int kEpiPlain = 0, kEpiSplit = 1, kEpiPlainFast = 2;  // epilogue variants (the kernel's EPI)
constexpr int kUnitRing = 4;        // unit indices in flight between the producer and the other roles
constexpr int kUnitReaders = 1 + 8;  // the MMA warp and one lane of each softmax warp (one more MMA warp with the score ring)
constexpr uint32_t kTmemCols = 512;
constexpr int kChunk = 64;          // bf16 elements per 128-byte chunk
constexpr uint32_t kChunkBytes = kBN * 128;  // one 128-byte column chunk of a 128-row tile
// Lazy-rescale threshold (log2 units).  P <= 2^32 is exact-range safe in bf16 (fp32 exponent
// range), and O and l accumulate in fp32 with room to spare (2^32 * |V| * S_k << 2^128); the
// relative precision of P, O and l does not depend on their scale.  A large threshold means the
// O rescale essentially only happens when a row's max jumps by more than 2^32.
constexpr float kTau = 32.0f;

__host__ __device__ constexpr uint32_t col_s(int t) { return static_cast<uint32_t>(t * 128); }
__host__ __device__ constexpr uint32_t col_o(int t) { return static_cast<uint32_t>(256 + t * 128); }

// One work unit: a 256-row query block of one (b, h) and one share of its key tiles.
struct Unit {
    int u, split;             // launch-order index (-1: no more units) and split-KV share
    int b, h, hk, r0;
    int j0, n_kv;             // the share's first key tile and its number of key tiles
    int as0, es0, as1, es1;   // key tiles [as_t, es_t) of the share that query tile t needs
};

struct Ctl {
    uint64_t full[kMaxSlots];
    uint64_t empty[kMaxSlots];
    uint64_t q_full;
    uint64_t q_empty;     // the unit's last Q K^T has read Q (the next unit's Q may be loaded)
    uint64_t s_full[2];   // scores of tile t ready (and every earlier MMA done)
    uint64_t p_full[2][2];  // the h-th P of tile t written, on barrier [t][h mod 2] (128 arrivals): with the
                            // score ring the softmax may hand over two P before the issuer takes the first
    uint64_t o_done[2];   // last P V of tile t done
    uint64_t s_read[2];   // score ring: softmax t has the scores in registers (128 arrivals)
    uint64_t o_ready[2][2];  // score ring: the c-th P V of tile t done, on barrier [t][c mod 2]
    uint64_t unit_full[kUnitRing];   // ring entry k written by the producer
    uint64_t unit_empty[kUnitRing];  // ring entry k read by every other role
    Unit unit[kUnitRing];            // decoded units (u = -1 once no CTA is left to take over)
    uint4 clc_resp;                  // response of the last launch-control request
    uint64_t clc_full;               // that response has landed
    uint64_t drain[2];  // a stopping MMA warp's products are done (one per MMA warp)
    uint64_t stall;
    uint32_t tmem_base;
    volatile uint32_t abort_flag;
};


// Units run over groups of `head_group` heads; inside a group, the heaviest query blocks first
// when work grows with the block index; the shares of one block are adjacent.
__device__ __forceinline__ Unit decode_unit(const AttnParams &p, int u) {
    Unit U;
    const int split = u % p.n_split;
    U.u = u;
    U.split = split;
    const int item = u / p.n_split;
    const int BH = p.B * p.H;
    const int per_group = p.head_group * p.n_qblocks;
    const int g = item / per_group;
    const int rr = item - g * per_group;
    const int g_heads = min(p.head_group, BH - g * p.head_group);
    const int slot_q = rr / g_heads;
    const int bh = g * p.head_group + (rr - slot_q * g_heads);
    const int qb = p.reverse_q ? (p.n_qblocks - 1 - slot_q) : slot_q;
    U.h = bh % p.H;
    U.b = bh / p.H;
    U.hk = U.h / p.kv_group;
    U.r0 = qb * kRows;
    // The union of both query tiles' key-tile ranges is contiguous (tile 1's first key never lies
    // past tile 0's last); it is cut into n_split contiguous shares.
    int a[2], e[2];
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        const int first = U.r0 + t * kBM;
        if (first >= p.S_q) {
            a[t] = 0;
            e[t] = 0;
        } else {
            band_tiles(p, first, min(first + kBM, p.S_q) - 1, kBN, &a[t], &e[t]);
        }
    }
    const bool has0 = e[0] > a[0], has1 = e[1] > a[1];
    const int A = has0 ? (has1 ? min(a[0], a[1]) : a[0]) : (has1 ? a[1] : 0);
    const int E = has0 ? (has1 ? max(e[0], e[1]) : e[0]) : (has1 ? e[1] : 0);
    const int n_item = E - A;
    const int per = (n_item + p.n_split - 1) / p.n_split;
    const int lo = min(split * per, n_item), hi = min(n_item, lo + per);
    U.j0 = A + lo;
    U.n_kv = hi - lo;
    int as[2], es[2];
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        as[t] = min(max(a[t] - U.j0, 0), U.n_kv);
        es[t] = min(max(e[t] - U.j0, 0), U.n_kv);
        if (es[t] <= as[t]) {
            as[t] = 0;
            es[t] = 0;
        }
    }
    U.as0 = as[0];
    U.es0 = es[0];
    U.as1 = as[1];
    U.es1 = es[1];
    return U;
}

// Invariants of a decoded unit, checked by the debug build before the unit's loads are issued.
__device__ __forceinline__ bool unit_valid(const AttnParams &p, const Unit &U) {
    const int tiles = (p.S_k + kBN - 1) / kBN;
    return U.b >= 0 && U.b < p.B && U.h >= 0 && U.h < p.H && U.hk == U.h / p.kv_group && U.r0 >= 0 &&
           U.r0 < p.S_q && U.r0 % kRows == 0 && U.split >= 0 && U.split < p.n_split && U.j0 >= 0 && U.n_kv >= 0 &&
           U.j0 + U.n_kv <= tiles && U.as0 >= 0 && U.as0 <= U.es0 && U.es0 <= U.n_kv && U.as1 >= 0 &&
           U.as1 <= U.es1 && U.es1 <= U.n_kv;
}

// The n-th unit this CTA works on, as the producer decoded and published it (u = -1: no more
// units); false on abort.  Called by a whole warp: lane 0 waits for the ring entry and releases it,
// every lane copies the unit (the producer decodes ahead, so readers spend no time on it).
__device__ __forceinline__ bool next_unit(Ctl &ctl, int n, Unit *out, const AttnParams &p, int lane) {
    const int k = n % kUnitRing;
    bool ok = true;
    if (lane == 0) ok = wait_bounded(smem_u32(&ctl.unit_full[k]), (n / kUnitRing) & 1, ctl.abort_flag, p);
    if (!__shfl_sync(0xffffffffu, ok, 0)) return false;
    __syncwarp();
    const volatile Unit *src = &ctl.unit[k];
    out->u = src->u;
    out->split = src->split;
    out->b = src->b;
    out->h = src->h;
    out->hk = src->hk;
    out->r0 = src->r0;
    out->j0 = src->j0;
    out->n_kv = src->n_kv;
    out->as0 = src->as0;
    out->es0 = src->es0;
    out->as1 = src->as1;
    out->es1 = src->es1;
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&ctl.unit_empty[k]));
    return true;
}

}  // namespace q2

// KQ: MMA K-steps (16 bf16 each) of Q K^T, D_qk rounded up: 2, 4, 6 or 8.
// RING: value widths up to 64, where TMEM holds a three-slot score ring per query tile (below), so the next
// key tile's scores are computed while the softmax works on the current ones.
// EPI: what the epilogue writes.  kEpiPlain: O (any alignment, any D_v, the log-sum-exp if asked for);
// kEpiSplit: the partial results of a key-range share, for the split-KV merge kernel; kEpiPlainFast: O only,
// 32-byte aligned rows and D_v a multiple of 16 (the common case, with no other store forms in the code).
// FOLD: the scale is positive and folds into the exponent; otherwise the scores are scaled first.
template <int KQ, bool RING, int EPI, bool FOLD>
__global__ void __launch_bounds__(q2::kThreads, 1)
    attn_fwd_bf16_2q_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                            const __grid_constant__ CUtensorMap tmV, const AttnParams p) {
    using namespace q2;
    constexpr int BN = kBN;
    __shared__ Ctl ctl;
    extern __shared__ uint8_t smem_raw[];

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    const int n_slots = p.stages;

    // ---- shared memory: Q tile 0, Q tile 1, then `n_slots` equal K/V slots
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const uint32_t q_tile_bytes = p.q_chunks * kChunkBytes;
    const uint32_t k_bytes = p.q_chunks * kChunkBytes;
    const uint32_t v_bytes = p.v_chunks * kChunkBytes;
    const uint32_t slot_bytes = max(k_bytes, v_bytes);
    const uint32_t sQ0 = base, sQ1 = base + q_tile_bytes;
    const uint32_t sSlot0 = base + 2 * q_tile_bytes;

    if (threadIdx.x == 0) {
        // with the score ring each query tile has its own MMA warp, and both release every slot and Q
        for (int s = 0; s < n_slots; ++s) {
            mbar_init(smem_u32(&ctl.full[s]), 1);
            mbar_init(smem_u32(&ctl.empty[s]), RING ? 2 : 1);
        }
        mbar_init(smem_u32(&ctl.q_full), 1);
        mbar_init(smem_u32(&ctl.q_empty), RING ? 2 : 1);
        for (int t = 0; t < 2; ++t) {
            mbar_init(smem_u32(&ctl.s_full[t]), 1);
            mbar_init(smem_u32(&ctl.p_full[t][0]), 128);
            mbar_init(smem_u32(&ctl.p_full[t][1]), 128);
            mbar_init(smem_u32(&ctl.o_done[t]), 1);
            mbar_init(smem_u32(&ctl.s_read[t]), 128);
            mbar_init(smem_u32(&ctl.o_ready[t][0]), 1);
            mbar_init(smem_u32(&ctl.o_ready[t][1]), 1);
        }
        for (int k = 0; k < kUnitRing; ++k) {
            mbar_init(smem_u32(&ctl.unit_full[k]), 1);
            mbar_init(smem_u32(&ctl.unit_empty[k]), kUnitReaders + (RING ? 1 : 0));
        }
        mbar_init(smem_u32(&ctl.drain[0]), 1);
        mbar_init(smem_u32(&ctl.drain[1]), 1);
        mbar_init(smem_u32(&ctl.stall), 1);
        mbar_init(smem_u32(&ctl.clc_full), 1);
        ctl.abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&ctl.tmem_base), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctl.tmem_base;

    if (warp < 4) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsControl));
    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            // loads i = 2j (K_j) and 2j + 1 (V_j) of a unit go to the ring's next slots
            int s = 0;
            uint32_t empty_phase = 0;  // bit s: parity of the next empty-phase of slot s to wait for
            int loads = 0, q_loads = 0;
            bool ok = true;
            bool clc_done = false;
            uint32_t clc_par = 0;
            for (int n = 0; ok; ++n) {
                // draw the next unit and publish it to the other roles
                const int k = n % kUnitRing;
                if (n >= kUnitRing) {
                    ok = wait_bounded(smem_u32(&ctl.unit_empty[k]), ((n / kUnitRing) - 1) & 1, ctl.abort_flag, p);
                    if (!ok) break;
                }
                // the CTA's own unit first, then those of CTAs whose launch this one cancels
                int u = -1;
                if (n == 0) {
                    u = static_cast<int>(blockIdx.x);
                } else if (!clc_done) {
                    mbar_arrive_expect_tx(smem_u32(&ctl.clc_full), 16);
                    clc_try_cancel(smem_u32(&ctl.clc_resp), smem_u32(&ctl.clc_full));
                    ok = wait_bounded(smem_u32(&ctl.clc_full), clc_par, ctl.abort_flag, p);
                    clc_par ^= 1u;
                    if (!ok) break;
                    u = clc_cancelled_x(smem_u32(&ctl.clc_resp));
                    if (u < 0) clc_done = true;  // no further request once one has found no CTA left
                }
                if (u >= p.n_units) u = -1;
                Unit U;
                if (u >= 0) {
                    U = decode_unit(p, u);
                    if (!VT_DEV_CHECK(!(p.flags & kFlagTestBounds) && unit_valid(p, U), ctl.abort_flag, p)) break;
                } else {
                    U.u = -1;
                    U.split = U.b = U.h = U.hk = U.r0 = U.j0 = U.n_kv = U.as0 = U.es0 = U.as1 = U.es1 = 0;
                }
                volatile Unit *dst_u = &ctl.unit[k];
                dst_u->u = U.u;
                dst_u->split = U.split;
                dst_u->b = U.b;
                dst_u->h = U.h;
                dst_u->hk = U.hk;
                dst_u->r0 = U.r0;
                dst_u->j0 = U.j0;
                dst_u->n_kv = U.n_kv;
                dst_u->as0 = U.as0;
                dst_u->es0 = U.es0;
                dst_u->as1 = U.as1;
                dst_u->es1 = U.es1;
                mbar_arrive(smem_u32(&ctl.unit_full[k]));
                if (u < 0) break;
                if (U.n_kv == 0) continue;
                // The unit's Q may only be loaded once the previous unit's last Q K^T has read the Q buffers;
                // fetch it into L2 now, so that the load after that point is an L2 hit.
                for (int t = 0; t < 2; ++t)
                    if ((t ? U.es1 > U.as1 : U.es0 > U.as0))
                        for (int c = 0; c < p.q_chunks; ++c) tma_prefetch_l2_4d(&tmQ, c * kChunk, U.r0 + t * kBM, U.h, U.b);
                if (q_loads > 0) {  // the previous unit's last Q K^T has read Q
                    ok = wait_bounded(smem_u32(&ctl.q_empty), (q_loads - 1) & 1, ctl.abort_flag, p);
                    if (!ok) break;
                }
                const bool load0 = U.es0 > U.as0, load1 = U.es1 > U.as1;  // Q tiles with work
                mbar_arrive_expect_tx(smem_u32(&ctl.q_full), (int(load0) + int(load1)) * q_tile_bytes);
                if (load0)
                    for (int c = 0; c < p.q_chunks; ++c)
                        tma_load_4d(sQ0 + c * kChunkBytes, &tmQ, smem_u32(&ctl.q_full), c * kChunk, U.r0, U.h, U.b);
                if (load1)
                    for (int c = 0; c < p.q_chunks; ++c)
                        tma_load_4d(sQ1 + c * kChunkBytes, &tmQ, smem_u32(&ctl.q_full), c * kChunk, U.r0 + kBM, U.h,
                                    U.b);
                ++q_loads;
                for (int i = 0; i < 2 * U.n_kv; ++i) {
                    if (loads >= n_slots) {
                        ok = wait_bounded(smem_u32(&ctl.empty[s]), (empty_phase >> s) & 1u, ctl.abort_flag, p);
                        empty_phase ^= 1u << s;
                        if (!ok) break;
                    }
                    const uint32_t dst = sSlot0 + s * slot_bytes;
                    const uint32_t bar = smem_u32(&ctl.full[s]);
                    const int j = i >> 1;
                    if (!VT_DEV_CHECK(s < n_slots && (U.j0 + j) * BN < p.S_k, ctl.abort_flag, p)) {
                        ok = false;
                        break;
                    }
                    if ((i & 1) == 0) {
                        mbar_arrive_expect_tx(bar, k_bytes);
                        for (int c = 0; c < p.q_chunks; ++c)
                            tma_load_4d(dst + c * kChunkBytes, &tmK, bar, c * kChunk, (U.j0 + j) * BN, U.hk, U.b);
                    } else {
                        mbar_arrive_expect_tx(bar, v_bytes);
                        for (int c = 0; c < p.v_chunks; ++c)
                            tma_load_4d(dst + c * kChunkBytes, &tmV, bar, c * kChunk, (U.j0 + j) * BN, U.hk, U.b);
                    }
                    ++loads;
                    if (++s == n_slots) s = 0;
                }
            }
            if (ctl.abort_flag) {
                // Let every copy this thread started land before the CTA's memory goes away: the
                // last Q load and the last min(loads, n_slots) slot loads, each on the phase it used.
                if (q_loads > 0) wait_drain(smem_u32(&ctl.q_full), (q_loads - 1) & 1, p);
                for (int k = max(0, loads - n_slots); k < loads; ++k)
                    wait_drain(smem_u32(&ctl.full[k % n_slots]), (k / n_slots) & 1, p);
            }
        }
    } else if (warp == 1 || (RING && warp == 2)) {
        // ------------------------------------------------------------ MMA issuer(s)
        // The whole warp runs this code with warp-uniform values and waits on every barrier; one lane,
        // chosen once by elect.sync, issues every MMA and commit (as a predicate, the warp stays converged).
        {
            const uint32_t idesc_qk = instr_desc(1, kBM, BN, 0);
            const uint32_t idesc_pv = instr_desc(1, kBM, p.n_pv, 1);
            // Descriptors as (low, high) words: offsets only move the low word (start address >> 4).
            const uint64_t qdesc0 = smem_desc_sw128(sQ0, 16, 1024);
            const uint64_t kdesc0 = smem_desc_sw128(sSlot0, 16, 1024);         // K slots: K-major
            const uint64_t vdesc0 = smem_desc_sw128(sSlot0, kChunkBytes, 1024);  // V slots: N-major
            const uint32_t q_hi = static_cast<uint32_t>(qdesc0 >> 32), k_hi = static_cast<uint32_t>(kdesc0 >> 32);
            const uint32_t v_hi = static_cast<uint32_t>(vdesc0 >> 32);
            const uint32_t q_lo0 = static_cast<uint32_t>(qdesc0);
            const uint32_t q_lo1 = q_lo0 + (q_tile_bytes >> 4);
            const uint32_t k_lo0 = static_cast<uint32_t>(kdesc0), v_lo0 = static_cast<uint32_t>(vdesc0);
            const uint32_t slot_step = slot_bytes >> 4;                          // descriptor units
            const uint32_t s_col0 = tmem + col_s(0), s_col1 = tmem + col_s(1);
            const uint32_t o_col0 = tmem + col_o(0), o_col1 = tmem + col_o(1);
            bool ok = true, any_mma = false;
            uint32_t full_phase = 0;  // bit s: parity of the next full-phase of slot s
            uint32_t h0 = 0, h1 = 0;          // P hand-overs of tile 0 / 1 taken so far
            uint32_t q_par = 0;               // parity of the next Q load
            // The lane that issues every MMA and commit of this warp, elected once: a commit tracks the MMAs
            // of the thread that issues it, so all of them come from this one lane.
            const uint32_t lead = elect_leader();

            // K/V slots are filled by TMA: the mbarrier's completed transaction count already makes
            // the bytes visible to the tensor core, so no tcgen05 fence is needed after this wait.
            // Every lane waits, so the issuing lane has itself observed the phase.
            auto wait1 = [&](uint32_t bar, uint32_t parity) -> bool {
                return __all_sync(0xffffffffu, wait_bounded(bar, parity, ctl.abort_flag, p)) != 0;
            };
            auto wait_full = [&](int s) -> bool {
                const bool r = wait1(smem_u32(&ctl.full[s]), (full_phase >> s) & 1u);
                full_phase ^= 1u << s;
                return r;
            };
            auto qk = [&](uint32_t d, uint32_t q_lo, uint32_t k_lo) {
#pragma unroll
                for (int kk = 0; kk < KQ; ++kk) {
                    const uint32_t off = (kk >> 2) * (kChunkBytes >> 4) + (kk & 3) * 2;
                    mma_ss_lead(d, q_lo + off, q_hi, k_lo + off, k_hi, idesc_qk, kk > 0, lead);
                }
            };
            auto pv = [&](uint32_t d, uint32_t a, uint32_t v_lo, uint32_t acc0) {
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk)
                    mma_ts_lead(d, a + kk * 8, v_lo + kk * 128, v_hi, idesc_pv, (acc0 | kk) ? 1u : 0u, lead);
            };

            if (p.flags & kFlagTestStall) ok = wait1(smem_u32(&ctl.stall), 0);  // test hook
            int ks = 0;  // slot of the next K tile (the ring runs on across units)
            if constexpr (RING) {
                // Score ring: tile t owns three 64-column TMEM slots from column 192 t, and O_t 64 columns from
                // 384 + 64 t.  Its g-th scores (counted over the CTA's life) sit in slots 0-1 for even g and
                // slots 1-2 for odd g, and their P overwrites slot 0 or slot 2, so the next scores never touch
                // the P still to be multiplied.  Warp 1 issues tile 0's products and warp 2 tile 1's, so one
                // tile's chain never waits behind the other's.  S_t = Q_t K_{j+1}^T is issued once softmax t
                // has read the scores of key tile j (s_read), ahead of P_t,j V_j; each P V commits
                // o_ready[t][c mod 2] (c: the tile's P V count), which the softmax consumes before it rescales
                // O_t and before the epilogue.  Both warps release every K/V slot and Q (two arrivals each).
                const int tm = warp - 1;
                const uint32_t s_reg = tmem + static_cast<uint32_t>(tm * 192);
                const uint32_t o_r = tmem + static_cast<uint32_t>(384 + tm * 64);
                const uint32_t q_lo = tm ? q_lo1 : q_lo0;
                auto s_at = [&](uint32_t gi) { return s_reg + ((gi & 1u) ? 64u : 0u); };
                auto p_at = [&](uint32_t gi) { return s_reg + ((gi & 1u) ? 128u : 0u); };
                uint32_t g = 0, cur = 0, nxt = 0, c = 0, h = 0, sr_par = 0;
                for (int n = 0; ok; ++n) {
                    Unit U;
                    if (!(ok = next_unit(ctl, n, &U, p, lane)) || U.u < 0) break;
                    const int n_kv = U.n_kv;
                    if (n_kv == 0) continue;
                    const int as = tm ? U.as1 : U.as0, es = tm ? U.es1 : U.es0;
                    // this tile takes part in key tile j when as <= j < es
                    auto act = [&](int j) { return j >= as && j < es; };
                    if (!(ok = wait1(smem_u32(&ctl.q_full), q_par))) break;
                    q_par ^= 1u;
                    if (!(ok = wait_full(ks))) break;
                    if (act(0)) {
                        cur = g++;
                        qk(s_at(cur), q_lo, k_lo0 + ks * slot_step);
                        mma_commit_lead(smem_u32(&ctl.s_full[tm]), lead);
                        any_mma = true;
                    }
                    if (es <= 1) mma_commit_lead(smem_u32(&ctl.q_empty), lead);  // this tile's last Q K^T (or none)
                    mma_commit_lead(smem_u32(&ctl.empty[ks]), lead);
                    for (int j = 0; ok && j < n_kv; ++j) {
                        const int vs = ks + 1 == n_slots ? 0 : ks + 1;  // slot of V_j
                        const int kn = vs + 1 == n_slots ? 0 : vs + 1;  // slot of K_{j+1} (or the next unit's K_0)
                        if (j + 1 < n_kv) {
                            // the next key tile's scores, as soon as the softmax holds the current ones
                            if (!(ok = wait_full(kn))) break;
                            if (act(j + 1)) {
                                if (act(j)) {
                                    if (!(ok = wait1(smem_u32(&ctl.s_read[tm]), sr_par))) break;
                                    sr_par ^= 1u;
                                    tc_fence_after();
                                }
                                nxt = g++;
                                qk(s_at(nxt), q_lo, k_lo0 + kn * slot_step);
                                mma_commit_lead(smem_u32(&ctl.s_full[tm]), lead);
                                any_mma = true;
                                if (j + 2 == es) mma_commit_lead(smem_u32(&ctl.q_empty), lead);  // this tile's last Q K^T
                            }
                            mma_commit_lead(smem_u32(&ctl.empty[kn]), lead);
                        }
                        if (!(ok = wait_full(vs))) break;
                        if (act(j)) {
                            if (!(ok = wait1(smem_u32(&ctl.p_full[tm][h & 1u]), (h >> 1) & 1u))) break;
                            ++h;
                            tc_fence_after();
                            pv(o_r, p_at(cur), v_lo0 + vs * slot_step, j > as);
                            mma_commit_lead(smem_u32(&ctl.o_ready[tm][c & 1u]), lead);
                            ++c;
                        }
                        if (act(j + 1)) cur = nxt;  // the scores (and P) of key tile j + 1
                        mma_commit_lead(smem_u32(&ctl.empty[vs]), lead);
                        ks = kn;
                    }
                }
            } else {
            for (int n = 0; ok; ++n) {
                Unit U;
                if (!(ok = next_unit(ctl, n, &U, p, lane)) || U.u < 0) break;
                const int n_kv = U.n_kv;
                if (n_kv == 0) continue;
                const int as0 = U.as0, es0 = U.es0, as1 = U.as1, es1 = U.es1;
                // query tile t takes part in key tile j when as_t <= j < es_t
                auto act0 = [&](int j) { return j >= as0 && j < es0; };
                auto act1 = [&](int j) { return j >= as1 && j < es1; };
                if (!(ok = wait1(smem_u32(&ctl.q_full), q_par))) break;
                q_par ^= 1u;
                if (!(ok = wait_full(ks))) break;
                {
                    const uint32_t k_lo = k_lo0 + ks * slot_step;
                    if (act0(0)) {
                        qk(s_col0, q_lo0, k_lo);
                        mma_commit_lead(smem_u32(&ctl.s_full[0]), lead);
                    }
                    if (act1(0)) {
                        qk(s_col1, q_lo1, k_lo);
                        mma_commit_lead(smem_u32(&ctl.s_full[1]), lead);
                    }
                    if (n_kv == 1) mma_commit_lead(smem_u32(&ctl.q_empty), lead);  // last Q K^T of the unit
                    mma_commit_lead(smem_u32(&ctl.empty[ks]), lead);
                    any_mma = true;
                }
                for (int j = 0; ok && j < n_kv; ++j) {
                    const int vs = ks + 1 == n_slots ? 0 : ks + 1;  // slot of V_j
                    const int kn = vs + 1 == n_slots ? 0 : vs + 1;  // slot of K_{j+1} (or the next unit's K_0)
                    const bool more = j + 1 < n_kv;
                    if (!(ok = wait_full(vs))) break;
                    const uint32_t v_lo = v_lo0 + vs * slot_step;
                    const uint32_t kn_lo = k_lo0 + kn * slot_step;
                    if (act0(j)) {
                        if (!(ok = wait1(smem_u32(&ctl.p_full[0][h0 & 1u]), (h0 >> 1) & 1u))) break;
                        ++h0;
                        tc_fence_after();
                        pv(o_col0, s_col0, v_lo, j > as0);
                    }
                    if (more && !(ok = wait_full(kn))) break;
                    if (act0(j + 1)) {
                        qk(s_col0, q_lo0, kn_lo);
                        mma_commit_lead(smem_u32(&ctl.s_full[0]), lead);
                    } else if (act0(j)) {
                        mma_commit_lead(smem_u32(&ctl.o_done[0]), lead);
                    }
                    if (act1(j)) {
                        if (!(ok = wait1(smem_u32(&ctl.p_full[1][h1 & 1u]), (h1 >> 1) & 1u))) break;
                        ++h1;
                        tc_fence_after();
                        pv(o_col1, s_col1, v_lo, j > as1);
                    }
                    mma_commit_lead(smem_u32(&ctl.empty[vs]), lead);
                    if (act1(j + 1)) {
                        qk(s_col1, q_lo1, kn_lo);
                        mma_commit_lead(smem_u32(&ctl.s_full[1]), lead);
                    } else if (act1(j)) {
                        mma_commit_lead(smem_u32(&ctl.o_done[1]), lead);
                    }
                    if (j + 2 == n_kv) mma_commit_lead(smem_u32(&ctl.q_empty), lead);  // last Q K^T of the unit
                    if (more) mma_commit_lead(smem_u32(&ctl.empty[kn]), lead);
                    ks = kn;
                }
            }
            }
            if (!ok && any_mma) {
                mma_commit_lead(smem_u32(&ctl.drain[warp - 1]), lead);
                if (lane == 0) wait_drain(smem_u32(&ctl.drain[warp - 1]), 0, p);
                __syncwarp();
            }
        }
    }
    } else {
        // ------------------------------------------------------------ softmax warpgroups
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmax));
        const int t = (warp - 4) >> 2;              // query tile of this warpgroup
        const int quad = warp & 3;                  // TMEM lane quadrant
        const int row = quad * 32 + lane;
        const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
        // score ring: slots from column 192 t, O_t at 384 + 64 t (see the MMA issuer); otherwise S_t and O_t
        const uint32_t s_base = tmem + lane_base + (RING ? static_cast<uint32_t>(t * 192) : col_s(t));
        const uint32_t o_addr = tmem + lane_base + (RING ? static_cast<uint32_t>(384 + t * 64) : col_o(t));
        // Non-positive scales are applied to the scores first (FOLD false), so the folded form below sees c > 0.
        const float c = FOLD ? p.scale_log2 : 1.0f;
        const float2 c2 = make_float2(c, c);
        uint32_t s_par = 0, o_par = 0;  // parities of the next scores and the next o_done of this tile
        uint32_t g = 0;                 // score ring: scores of this tile seen over the CTA's life
        uint32_t handed = 0;            // P hand-overs of this tile over the CTA's life
        uint32_t pv_handed = 0, pv_seen = 0;  // score ring: P hand-overs, and P V completions consumed
        bool ok = true;
        // score ring: consume the completion of the oldest P V not yet consumed
        auto wait_pv = [&]() -> bool {
            const bool r = wait_bounded(smem_u32(&ctl.o_ready[t][pv_seen & 1u]), (pv_seen >> 1) & 1u, ctl.abort_flag, p);
            ++pv_seen;
            return __all_sync(0xffffffffu, r) != 0;
        };

        for (int n = 0; ok; ++n) {
            Unit U;
            if (!(ok = next_unit(ctl, n, &U, p, lane)) || U.u < 0) break;
            const int tile_row0 = U.r0 + t * kBM;
            const int q_row = tile_row0 + row;
            const int as_my = t ? U.as1 : U.as0;
            const int n_my = (t ? U.es1 : U.es0) - as_my;
            // this row's allowed keys [key_lo, key_hi); a key tile starting below mask_lo or ending past
            // mask_hi cuts some row's range and is masked (the same decision for the whole warpgroup)
            const int key_lo = band_key_lo(p, q_row), key_hi = band_key_hi(p, q_row);
            const int mask_lo = band_key_lo(p, min(tile_row0 + kBM, p.S_q) - 1);
            const int mask_hi = band_key_hi(p, tile_row0);
            float m_used = -INFINITY;  // reference max (log2 units) of O_t and l
            float l = 0.0f;
            float l_fix = 0.0f;        // bf16 rounding of each tile's largest P, relative to m_used

            for (int j = 0; j < n_my; ++j) {
                ok = wait_bounded(smem_u32(&ctl.s_full[t]), s_par, ctl.abort_flag, p);
                s_par ^= 1u;
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                tc_fence_after();
                const uint32_t s_addr = s_base + ((RING && (g & 1u)) ? 64u : 0u);   // scores
                const uint32_t p_addr = s_base + ((RING && (g & 1u)) ? 128u : 0u);  // P over them
                uint32_t sr[BN];
                #pragma unroll
                for (int cc = 0; cc < BN / 32; ++cc) tmem_ld32(s_addr + cc * 32, sr + cc * 32);
                tmem_wait_ld();
                if (RING && j + 1 < n_my) {  // the next scores may now be written over these
                    tc_fence_before();
                    mbar_arrive(smem_u32(&ctl.s_read[t]));
                }
                float s[BN];
                #pragma unroll
                for (int k = 0; k < BN; ++k) s[k] = __uint_as_float(sr[k]);
                if constexpr (!FOLD) {
                    #pragma unroll
                    for (int k = 0; k < BN; ++k) s[k] *= p.scale_log2;
                }
                const int k0 = (U.j0 + as_my + j) * BN;
                if (k0 < mask_lo || k0 + BN > mask_hi) {
                    #pragma unroll
                    for (int k = 0; k < BN; ++k)
                        if (k0 + k < key_lo || k0 + k >= key_hi) s[k] = -INFINITY;
                }
                float mx0 = fmax3(s[0], s[1], s[2]), mx1 = fmax3(s[3], s[4], s[5]);
                float mx2 = fmax3(s[6], s[7], s[8]), mx3 = fmax3(s[9], s[10], s[11]);
                #pragma unroll
                for (int k = 12; k < BN - 4; k += 8) {
                    mx0 = fmax3(mx0, s[k], s[k + 1]);
                    mx1 = fmax3(mx1, s[k + 2], s[k + 3]);
                    mx2 = fmax3(mx2, s[k + 4], s[k + 5]);
                    mx3 = fmax3(mx3, s[k + 6], s[k + 7]);
                }
                mx0 = fmax3(mx0, s[BN - 4], s[BN - 3]);
                mx1 = fmax3(mx1, s[BN - 2], s[BN - 1]);
                const float m_raw = fmax3(fmaxf(mx0, mx1), mx2, mx3);
                const float m_tile = m_raw * c;  // c > 0: -inf stays -inf
                const float m_new = fmaxf(m_used, m_tile);
                // Lazy rescale: keep the old reference unless the max grew by more than tau.
                const bool resc = (m_used == -INFINITY) ? (m_new != -INFINITY) : (m_new - m_used > kTau);
                float alpha = 1.0f;
                if (resc) {
                    alpha = (m_used == -INFINITY) ? 0.0f : ex2(m_used - m_new);
                    l *= alpha;
                    l_fix *= alpha;
                    m_used = m_new;
                }
                const float m_ref = (m_used == -INFINITY) ? 0.0f : m_used;
                const float2 nm2 = make_float2(-m_ref, -m_ref);
                // P V multiplies P rounded to bf16, while l adds the fp32 values.  The tile's largest P,
                // formed exactly as below, gives its rounding error to l_fix, and O is divided by l + l_fix:
                // a key that dominates its row then carries the same weight in both (exact when one key
                // dominates).  The log-sum-exp uses l alone.
                const float p_top = ex2(__fmaf_rn(m_raw, c, -m_ref));
                l_fix += __uint_as_float(pack_bf16x2(p_top, 0.0f) << 16) - p_top;
                float2 acc0 = make_float2(0.f, 0.f), acc1 = acc0;
                // P_t,j over S_t,j (bf16 pairs): each 32-score chunk goes to TMEM as 16 columns as
                // soon as it is exponentiated, which keeps the live registers near the 128 scores.
                #pragma unroll
                for (int cc = 0; cc < BN; cc += 32) {
                    uint32_t pk[16];
                    #pragma unroll
                    for (int k = 0; k < 32; k += 4) {
                        const float2 x0 = __ffma2_rn(make_float2(s[cc + k], s[cc + k + 1]), c2, nm2);
                        const float2 x1 = __ffma2_rn(make_float2(s[cc + k + 2], s[cc + k + 3]), c2, nm2);
                        const float2 e0 = make_float2(ex2(x0.x), ex2(x0.y));
                        const float2 e1 = make_float2(ex2(x1.x), ex2(x1.y));
                        acc0 = __fadd2_rn(acc0, e0);
                        acc1 = __fadd2_rn(acc1, e1);
                        pk[k / 2] = pack_bf16x2(e0.x, e0.y);
                        pk[k / 2 + 1] = pack_bf16x2(e1.x, e1.y);
                    }
                    tmem_st16(p_addr + cc / 2, pk);
                }
                l += (acc0.x + acc0.y) + (acc1.x + acc1.y);
                // O_t *= alpha where the reference moved (after the scores are dead, to keep registers
                // low).  The scores just read were committed after P_t,j-1 V_j-1, so O_t holds its final
                // value for tile j-1 and no MMA touches it now.
                if (j > 0 && __any_sync(0xffffffffu, resc)) {
                    if (RING) {  // O_t must hold every P V handed over so far
                        bool w = true;
                        while (w && pv_seen < pv_handed) w = wait_pv();
                        if (!(ok = w)) break;
                        tc_fence_after();
                    }
                    for (int cc = 0; cc < p.n_pv; cc += 32) {
                        uint32_t o[32];
                        tmem_ld32(o_addr + cc, o);
                        tmem_wait_ld();
                        #pragma unroll
                        for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
                        tmem_st32(o_addr + cc, o);
                    }
                }
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(smem_u32(&ctl.p_full[t][handed & 1u]));
                ++handed;
                if (RING) {
                    ++pv_handed;
                    ++g;
                    if (pv_handed - pv_seen >= 2 && !(ok = wait_pv())) break;  // at most one P V outstanding
                }
            }

            if (ok && n_my > 0) {
                if (RING) {
                    while (ok && pv_seen < pv_handed) ok = wait_pv();
                } else {
                    ok = wait_bounded(smem_u32(&ctl.o_done[t]), o_par, ctl.abort_flag, p);
                    o_par ^= 1u;
                    ok = __all_sync(0xffffffffu, ok);
                }
            }
            const bool row_ok = q_row < p.S_q;
            if (ok && EPI != kEpiSplit) {
                // ------------------------------------------------------------ epilogue: O = O_t / l
                // A row with no allowed key (l = 0, or no key tile at all) is written as 0.
                if (n_my > 0) tc_fence_after();
                const float inv_l = l > 0.0f ? 1.0f / (l + l_fix) : 0.0f;
                uint8_t *orow = reinterpret_cast<uint8_t *>(p.O) +
                                (static_cast<long long>(U.b) * p.o_sb + static_cast<long long>(U.h) * p.o_sh +
                                 static_cast<long long>(q_row) * p.o_ss) * 2;
                for (int cc = 0; cc < p.n_pv; cc += 16) {
                    uint32_t o[16];
                    if (n_my > 0) {
                        tmem_ld16(o_addr + cc, o);
                        tmem_wait_ld();
                    } else {
                        #pragma unroll
                        for (int k = 0; k < 16; ++k) o[k] = 0u;
                    }
                    if (!row_ok) continue;
                    uint32_t w[8];
                    #pragma unroll
                    for (int k = 0; k < 8; ++k)
                        w[k] = pack_bf16x2(__uint_as_float(o[2 * k]) * inv_l, __uint_as_float(o[2 * k + 1]) * inv_l);
                    if constexpr (EPI == kEpiPlainFast) {
                        st_global_v8(orow + cc * 2, w);  // one 32-byte store per 16 columns
                    } else if (cc + 16 <= p.D_v) {
                        if (p.o_vec32) {  // half as many store instructions, each a full 32-byte sector
                            st_global_v8(orow + cc * 2, w);
                        } else {
                            uint4 *dst = reinterpret_cast<uint4 *>(orow + cc * 2);
                            dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
                            dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
                        }
                    } else {
                        uint16_t *dst = reinterpret_cast<uint16_t *>(orow) + cc;
                        #pragma unroll
                        for (int k = 0; k < 16; ++k)
                            if (cc + k < p.D_v) dst[k] = static_cast<uint16_t>((w[k >> 1] >> ((k & 1) * 16)) & 0xFFFFu);
                    }
                }
                if (EPI == kEpiPlain && p.lse && row_ok)
                    p.lse[(static_cast<long long>(U.b) * p.H + U.h) * p.S_q + q_row] = lse_from(m_used, l);
            } else if (ok && EPI == kEpiSplit) {
                // ------------------------------------------------------------ epilogue: partial O, m, l
                // Unnormalised O_t with its reference max m (log2 units) and sum l; a share with no
                // key tile for this query tile writes the empty partial (m = -inf, l = 0, O = 0).
                const long long row_lin = (static_cast<long long>(U.b) * p.H + U.h) * p.S_q + q_row;
                const long long part = static_cast<long long>(U.split) * p.B * p.H * p.S_q + row_lin;
                float *orow = p.part_o + part * p.D_v;
                if (n_my > 0) tc_fence_after();
                for (int cc = 0; cc < p.n_pv; cc += 16) {
                    uint32_t o[16];
                    if (n_my > 0) {
                        tmem_ld16(o_addr + cc, o);
                        tmem_wait_ld();
                    } else {
                        #pragma unroll
                        for (int k = 0; k < 16; ++k) o[k] = 0u;
                    }
                    if (!row_ok) continue;
                    if (cc + 16 <= p.D_v) {
                        float4 *dst = reinterpret_cast<float4 *>(orow + cc);
                        #pragma unroll
                        for (int k = 0; k < 4; ++k)
                            dst[k] = make_float4(__uint_as_float(o[4 * k]), __uint_as_float(o[4 * k + 1]),
                                                 __uint_as_float(o[4 * k + 2]), __uint_as_float(o[4 * k + 3]));
                    } else {
                        #pragma unroll
                        for (int k = 0; k < 16; ++k)
                            if (cc + k < p.D_v) orow[cc + k] = __uint_as_float(o[k]);
                    }
                }
                if (row_ok) {
                    p.part_m[part] = n_my > 0 ? m_used : -INFINITY;
                    p.part_l[part] = n_my > 0 ? l : 0.0f;
                    p.part_c[part] = n_my > 0 ? l_fix : 0.0f;
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace vt
