// Attention forward of an MHA layer with the max logit taken along: the
// softmax inputs s_ij = q_i . k_j are computed anyway, so S_max^h of the
// MuonClip step ("Kimi K2" section 2.1 and the K2 notes: the clip uses the
// max logit of this step and leaves the forward unchanged) costs one max per
// logit on top of O = softmax(Q K^T / sqrt(dh)) V.
//
// This kernel runs dh = 64; dh = 128 runs on the MLA kernel below with two
// 64-wide blocks per logit (P over the S columns in TMEM).
//
// Work item = (sequence b, head h, pair of 128-query tiles); one persistent
// CTA per SM; items in bands of (b, h) pairs dealt in snake-ordered rounds
// (as in the scan).  Per 128-key block j of an item:
//   warp 0      TMA: both Q tiles once, then the K_j tiles (128 keys x dh)
//               into a K ring
//   warp 2      TMA: the V_j tiles into a V ring
//   warp 1      tcgen05.mma S_t = Q_t K_j^T for both tiles into two
//               128 x 128 fp32 TMEM tiles; once P_t is ready, O_t += P_t V
//               into the tile's 128 x dh fp32 TMEM accumulator (V MN-major
//               as stored; P_t from TMEM)
//   warpgroups 1, 2   one query row per thread of tile 0 / tile 1: S_t from
//               TMEM, the raw row max (for S_max), the running softmax max m
//               and sum l, O_t rescaled in TMEM when m moves, P_t = 2^(s - m)
//               as bf16; at the end of the item O_t / l as bf16, and per
//               warp S = max / sqrt(dh) max-merged into S_max[h] (and
//               S_max[b, h]) by one integer atomic each, as in the scan
#include "common.cuh"
#include "internal.h"

namespace mc {

// 384 threads, three warpgroups:
//   warpgroup 0  warp 0: TMA of Q (both tiles) and K; warp 1: TMEM owner and
//                MMA issuer; warp 2: TMA of V; warp 3 idle
//   warpgroup 1  softmax and output of query tile 0 (one row per thread)
//   warpgroup 2  softmax and output of query tile 1
// Registers move from warpgroup 0 to the softmax warpgroups with setmaxnreg
// (128 x 96 + 256 x 200 = 63488 <= 384 threads x 168 at launch); each
// warpgroup's branch starts with its setmaxnreg, so the compiler allocates
// the softmax code with the larger budget (128 logits per thread stay in
// registers, and P is packed for TMEM).
constexpr int kAttnThreads = 384;
constexpr int kAttnRegsLow = 96, kAttnRegsHigh = 200;
static_assert(128 * kAttnRegsLow + 256 * kAttnRegsHigh <= kAttnThreads * (65536 / kAttnThreads / 8 * 8),
              "register split");
constexpr int kAttnBlk = 128;          // queries per tile, keys per key block
constexpr int kAttnMaxStages = 4;
constexpr int kAttnTile = 16384;       // 128 rows x 64 bf16 (one 128-byte-swizzled block)
constexpr int kAttnRing = 224 * 1024;  // Q of two tiles, then the K and V rings
constexpr int kAttnSmem = 1024 + 1024 + kAttnRing;

struct AttnParams {
    CUtensorMap tmQ, tmK, tmV;  // {H*dh, T, B} bf16, box {64, 128}
    CUtensorMap tmKR;           // MLA: the shared k^R {kr_ld, T, B}, box {64, 128}
    int kr_col;
    int B, T, H, dh, causal;
    int n_it, n_pair, total_items, band, kst, vst;
    __nv_bfloat16* o;
    long long ld;               // H * dh: row stride of q, k, v and o
    float scale_log2;           // log2(e) / sqrt(dh)
    float sqrt_d;
    float* s_max;
    float* s_bh;
    unsigned* status;
};

struct AttnSmemTail {
    uint64_t kfull[kAttnMaxStages], kempty[kAttnMaxStages];
    uint64_t vfull[kAttnMaxStages], vempty[kAttnMaxStages];
    uint64_t qfull, qempty;
    uint64_t sfull[2], sempty[2];  // per query tile
    uint64_t pfull[2];
    uint64_t oready[2];  // one phase per P.V product of the tile
    uint64_t oempty[2];  // the tile's output of an item has been read from TMEM
    uint64_t drain;
    uint32_t tmem_base;
    int abort_flag;
};

// 2^x with the hardware approximation (relative error about 2^-22, far below
// the bf16 rounding of the softmax weights; tiny results flush to zero)
MC_D float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Item i -> (b, h, tile pair g) and the key blocks of its two query tiles
// 2g and 2g + 1 (0 when the tile lies past the sequence).
MC_D void attn_item(const AttnParams& P, int i, int& b, int& h, int& g, int (&njb)[2]) {
    const int BH = P.B * P.H;
    const int per_band = P.band * P.n_pair;
    const int band = i / per_band;
    const int w = i - band * per_band;
    const int pairs = min(P.band, BH - band * P.band);
    const int grp = w / pairs;
    const int bh = band * P.band + (w - grp * pairs);
    g = P.causal ? (P.n_pair - 1 - grp) : grp;  // heaviest causal pairs first
    b = bh / P.H;
    h = bh - b * P.H;
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        const int it = 2 * g + t;
        const int row_end = min(P.T, (it + 1) * kAttnBlk);
        njb[t] = it >= P.n_it ? 0
                 : P.causal   ? (row_end - 1) / kAttnBlk + 1
                              : (P.T + kAttnBlk - 1) / kAttnBlk;
    }
}

MC_D int attn_round_item(int r) {
    const int c = (r & 1) ? (int)(gridDim.x - 1 - blockIdx.x) : (int)blockIdx.x;
    return r * (int)gridDim.x + c;
}

// The MMA warp shares its SM sub-partition with two softmax warps, so its
// issue path is kept short: descriptors are formed once per tile or stage
// and a K step only adds a constant to the 16-byte address field.
// S_t = Q_t K^T at dh = 64: K-major Q and K, one 64-wide block, 4 steps
MC_D void issue_s(uint32_t d_tmem, uint64_t qd, uint64_t kd, uint32_t idesc) {
#pragma unroll
    for (int k = 0; k < 4; ++k) umma_bf16(d_tmem, qd + (uint64_t)(k * 2), kd + (uint64_t)(k * 2), idesc, k != 0);
}

// O_t (+)= P_t V with P_t in TMEM (one row per lane, two bf16 keys per
// 32-bit column, 64 columns for 128 keys) as the A operand, 8 columns per
// K step; V MN-major (2 KB per K step)
MC_D void issue_pv_tmem_a(uint32_t d_tmem, uint32_t p_tmem, uint64_t vd, uint32_t idesc, bool acc) {
#pragma unroll
    for (int k = 0; k < kAttnBlk / 16; ++k) {
        const uint32_t en = (acc || k != 0) ? 1u : 0u;
        asm volatile(
            "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
            "r"(p_tmem + (uint32_t)(k * 8)), "l"(vd + (uint64_t)(k * (2048 >> 4))), "r"(idesc), "r"(en));
    }
}

template <uint32_t N>
MC_D void setmaxnreg_inc() { asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N)); }
template <uint32_t N>
MC_D void setmaxnreg_dec() { asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N)); }

__global__ void __launch_bounds__(kAttnThreads, 1) attn_kernel(const __grid_constant__ AttnParams P) {
    constexpr int DH = 64;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    static_assert(sizeof(AttnSmemTail) <= 1024, "tail");
    AttnSmemTail* tail = reinterpret_cast<AttnSmemTail*>(smem);
    uint8_t* sQ = smem + 1024;             // tile t: block t
    uint8_t* sK = sQ + 2 * kAttnTile;      // stage s: one block
    uint8_t* sV = sK + P.kst * kAttnTile;
    volatile int* abort_flag = &tail->abort_flag;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t blk_bytes = (uint32_t)kAttnTile;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kAttnMaxStages; ++s) {
            mbar_init(&tail->kfull[s], 1);
            mbar_init(&tail->kempty[s], 1);
            mbar_init(&tail->vfull[s], 1);
            mbar_init(&tail->vempty[s], 1);
        }
        mbar_init(&tail->qfull, 1);
        mbar_init(&tail->qempty, 1);
        for (int t = 0; t < 2; ++t) {
            mbar_init(&tail->sfull[t], 1);
            mbar_init(&tail->sempty[t], 4);
            mbar_init(&tail->pfull[t], 4);
            mbar_init(&tail->oready[t], 1);
            mbar_init(&tail->oempty[t], 4);
        }
        mbar_init(&tail->drain, 1);
        tail->abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&P.tmQ);
        tma_prefetch_desc(&P.tmK);
        tma_prefetch_desc(&P.tmV);
    }
    if (warp == 1) {
        tmem_alloc(&tail->tmem_base, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = tail->tmem_base;  // S tiles at columns 0 and 128, O tiles from 256
    pdl_wait();

    if (warp < 4) {
    setmaxnreg_dec<kAttnRegsLow>();
    if (warp == 0 || warp == 2) {
        // ---------------- TMA producers: Q and K (warp 0), V (warp 2) ----------------
        if (lane == 0) {
            const bool is_k = warp == 0;
            const int nst = is_k ? P.kst : P.vst;
            uint64_t* full = is_k ? tail->kfull : tail->vfull;
            uint64_t* empty = is_k ? tail->kempty : tail->vempty;
            uint8_t* ring = is_k ? sK : sV;
            const CUtensorMap* tm = is_k ? &P.tmK : &P.tmV;
            int stage = 0;
            uint32_t phase = 0;
            uint32_t issued[kAttnMaxStages] = {0, 0, 0, 0};
            uint32_t n = 0;
            bool ok = true;
            for (int r = 0, i = attn_round_item(0); i < P.total_items && ok; i = attn_round_item(++r), ++n) {
                int b, h, g, njb[2];
                attn_item(P, i, b, h, g, njb);
                if (is_k) {
                    // both Q tiles (the second may lie past the sequence: zeros)
                    if (!mbar_wait(&tail->qempty, (n & 1) ^ 1, abort_flag, P.status)) break;
                    mbar_arrive_expect_tx(&tail->qfull, 2 * blk_bytes);
                    for (int t = 0; t < 2; ++t)
                        tma_load_3d(sQ + t * kAttnTile, &P.tmQ, &tail->qfull, h * DH, (2 * g + t) * kAttnBlk, b);
                }
                const int nj = max(njb[0], njb[1]);
                for (int j = 0; j < nj; ++j) {
                    if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag, P.status)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&full[stage], blk_bytes);
                    tma_load_3d(ring + stage * kAttnTile, tm, &full[stage], h * DH, j * kAttnBlk, b);
                    ++issued[stage];
                    if (++stage == nst) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
            }
            // the copies still in flight land before exit
            volatile int never = 0;
            for (int s = 0; s < nst; ++s)
                if (issued[s]) mbar_wait(&full[s], (issued[s] - 1) & 1, &never, P.status);
            if (is_k && n) mbar_wait(&tail->qfull, (n - 1) & 1, &never, P.status);
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        const uint32_t idesc_s = idesc_f16kind(kAttnBlk, kAttnBlk, 0, 0);  // S = Q K^T, K-major K
        const uint32_t idesc_o = idesc_f16kind(kAttnBlk, DH, 1, 0);      // O += P V, MN-major V
        int ks = 0, vs = 0;
        uint32_t kph = 0, vph = 0;
        uint32_t sc[2] = {0, 0}, pc[2] = {0, 0}, no[2] = {0, 0}, n = 0;
        bool ok = true;
        int njb[2];
        // descriptors of tile 0 / ring stage 0; tile 1 and stage s add a
        // multiple of the block size (in 16-byte units) to the address field
        const uint64_t qdesc0 = sw128_desc(smem_u32(sQ), 16, 1024);
        const uint64_t kdesc0 = sw128_desc(smem_u32(sK), 16, 1024);
        const uint64_t vdesc0 = sw128_desc(smem_u32(sV), kAttnTile, 1024);
        const uint64_t blk16 = (uint64_t)kAttnTile >> 4;  // one stage or one Q tile
        // O_t += P_t V_jj for both tiles that use key block jj; the first
        // product of an item overwrites O_t once the previous output is read
        // Each pair of products waits for both tiles' barriers first and is
        // then issued back to back: this thread's control steps are slow on a
        // sub-partition shared with two softmax warps, and the tensor pipe
        // drains during every step between two batches of MMAs.
        auto pv = [&](int jj) {
            if (!mbar_wait(&tail->vfull[vs], vph, abort_flag, P.status)) return false;
            for (int t = 0; t < 2; ++t) {
                if (jj >= njb[t]) continue;
                if (jj == 0 && !mbar_wait(&tail->oempty[t], (no[t] & 1) ^ 1, abort_flag, P.status)) return false;
                if (!mbar_wait(&tail->pfull[t], pc[t] & 1, abort_flag, P.status)) return false;
            }
            tc_fence_after();
            if (lane == 0) {
                for (int t = 0; t < 2; ++t) {
                    if (jj >= njb[t]) continue;
                    // P_t in TMEM after O0 and O1
                    issue_pv_tmem_a(tmem_base + 256 + t * DH, tmem_base + 256 + 2 * DH + t * (kAttnBlk / 2),
                                    vdesc0 + (uint64_t)vs * blk16, idesc_o, jj != 0);
                    umma_commit(&tail->oready[t]);
                }
                umma_commit(&tail->vempty[vs]);  // V_jj consumed by both tiles
            }
            __syncwarp();
            for (int t = 0; t < 2; ++t) {
                if (jj >= njb[t]) continue;
                ++pc[t];
                if (jj == njb[t] - 1) ++no[t];
            }
            if (++vs == P.vst) {
                vs = 0;
                vph ^= 1;
            }
            return true;
        };
        for (int r = 0, i = attn_round_item(0); i < P.total_items && ok; i = attn_round_item(++r), ++n) {
            int b, h, g;
            attn_item(P, i, b, h, g, njb);
            const int nj = max(njb[0], njb[1]);
            if (!mbar_wait(&tail->qfull, n & 1, abort_flag, P.status)) break;
            for (int j = 0; j < nj && ok; ++j) {
                // S_t = Q_t K_j^T for the tiles that use key block j
                if (!mbar_wait(&tail->kfull[ks], kph, abort_flag, P.status)) {
                    ok = false;
                    break;
                }
                for (int t = 0; t < 2 && ok; ++t) {
                    if (j >= njb[t]) continue;
                    if (!mbar_wait(&tail->sempty[t], (sc[t] & 1) ^ 1, abort_flag, P.status)) ok = false;
                }
                if (!ok) break;
                tc_fence_after();
                if (lane == 0) {
                    for (int t = 0; t < 2; ++t) {
                        if (j >= njb[t]) continue;
                        const uint64_t qd = qdesc0 + (uint64_t)t * blk16, kd = kdesc0 + (uint64_t)ks * blk16;
                        issue_s(tmem_base + t * kAttnBlk, qd, kd, idesc_s);
                        umma_commit(&tail->sfull[t]);
                    }
                    umma_commit(&tail->kempty[ks]);                // K_j consumed
                    if (j == nj - 1) umma_commit(&tail->qempty);  // the item's last use of Q
                }
                __syncwarp();
                for (int t = 0; t < 2; ++t)
                    if (j < njb[t]) ++sc[t];
                if (++ks == P.kst) {
                    ks = 0;
                    kph ^= 1;
                }
                // O_t += P_t V_{j-1} while the softmax works on S_j
                if (j >= 1 && !pv(j - 1)) {
                    ok = false;
                    break;
                }
            }
            if (!ok) break;
            if (!pv(nj - 1)) break;
        }
        if (lane == 0) umma_commit(&tail->drain);
        __syncwarp();
        volatile int never = 0;
        mbar_wait(&tail->drain, 0, &never, P.status);
    }
    } else {
        setmaxnreg_inc<kAttnRegsHigh>();
        // ---------------- softmax and output: tile t = warpgroup - 1 ----------------
        const int t = warp >= 8 ? 1 : 0;
        const int quarter = warp & 3;        // TMEM lanes 32 q .. 32 q + 31
        const int lr = quarter * 32 + lane;  // row of the tile
        const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
        const uint32_t tS = tmem_base + lane_base + t * kAttnBlk;
        const uint32_t tO = tmem_base + lane_base + 256 + t * DH;
        const uint32_t tP = tmem_base + lane_base + 256 + 2 * DH + t * (kAttnBlk / 2);
        uint32_t sc = 0, pc = 0;
        bool ok = true;
        for (int r = 0, i = attn_round_item(0); i < P.total_items && ok; i = attn_round_item(++r)) {
            int b, h, g, njb[2];
            attn_item(P, i, b, h, g, njb);
            const int nj = njb[t];
            if (nj == 0) continue;  // the tile lies past the sequence
            const int it = 2 * g + t;
            const int row = it * kAttnBlk + lr;
            const bool row_ok = row < P.T;
            float m = -INFINITY, l = 0.f, m_raw = -INFINITY;
            for (int j = 0; j < nj && ok; ++j) {
                if (!mbar_wait(&tail->sfull[t], sc & 1, abort_flag, P.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                float v[kAttnBlk];
                uint32_t* vu = reinterpret_cast<uint32_t*>(v);
#pragma unroll
                for (int c = 0; c < kAttnBlk / 32; ++c) tmem_ld32(tS + c * 32, vu + c * 32);
                tmem_ld_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&tail->sempty[t]);
                ++sc;
                // mask (keys past T; keys after the row when causal; rows past T)
                const int key0 = j * kAttnBlk;
                const bool full = (it + 1) * kAttnBlk <= P.T && key0 + kAttnBlk <= P.T &&
                                  (!P.causal || key0 + kAttnBlk - 1 <= it * kAttnBlk);
                if (!full) {
                    const int lim = !row_ok ? 0 : (P.causal ? min(row + 1, P.T) : P.T);  // keys < lim
#pragma unroll
                    for (int e = 0; e < kAttnBlk; ++e)
                        if (key0 + e >= lim) v[e] = -INFINITY;
                }
                // four independent max chains (the row max), then one
                float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                for (int e = 0; e < kAttnBlk; e += 8)
#pragma unroll
                    for (int c = 0; c < 4; ++c) m4[c] = max3_nan(m4[c], v[e + 2 * c], v[e + 2 * c + 1]);
                const float mb = max_nan(max_nan(m4[0], m4[1]), max_nan(m4[2], m4[3]));
                m_raw = max_nan(m_raw, mb);
                // softmax in base 2: x = s log2(e) / sqrt(dh).  P, O and l are
                // relative to the reference max m, which moves (and O with it)
                // only when the row max exceeds it by more than 8: the weights
                // stay below 2^8 and most blocks skip the rescale.
                const float mx = mb * P.scale_log2;
                const float m_new = !row_ok ? 0.f : (mx > m + 8.f || m == -INFINITY) ? fmaxf(m, mx) : m;
                const float alpha = row_ok && m_new != m ? ex2_approx(m - m_new) : 1.f;
                // pairs of logits through the packed fp32 FMA and add of
                // sm_100+; logit e goes to partial sum e mod 8
                const float2 sc2 = make_float2(P.scale_log2, P.scale_log2), nm2 = make_float2(-m_new, -m_new);
                float2 ls[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                                make_float2(0.f, 0.f)};
#pragma unroll
                for (int e = 0; e < kAttnBlk; e += 2) {
                    const float2 x = __ffma2_rn(make_float2(v[e], v[e + 1]), sc2, nm2);
                    const float p0 = row_ok ? ex2_approx(x.x) : 0.f, p1 = row_ok ? ex2_approx(x.y) : 0.f;
                    v[e] = p0;
                    v[e + 1] = p1;
                    ls[(e >> 1) & 3] = __fadd2_rn(ls[(e >> 1) & 3], make_float2(p0, p1));
                }
                const float lsum = ((ls[0].x + ls[0].y) + (ls[1].x + ls[1].y)) + ((ls[2].x + ls[2].y) + (ls[3].x + ls[3].y));
                l = __fmaf_rn(l, alpha, lsum);
                m = m_new;
                if (j >= 1) {
                    // O_t and the P tile are free once P_{j-1} V_{j-1} is done
                    if (!mbar_wait(&tail->oready[t], (pc - 1) & 1, abort_flag, P.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    if (__any_sync(0xFFFFFFFFu, alpha != 1.f)) {
                        #pragma unroll 1
                        for (int c = 0; c < DH / 32; ++c) {
                            uint32_t o[32];
                            tmem_ld32(tO + c * 32, o);
                            tmem_ld_wait();
#pragma unroll
                            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                            tmem_st32(tO + c * 32, o);
                        }
                        tmem_st_wait();
                    }
                }
                // P_j as bf16 pairs into this row's 64 TMEM columns (the A
                // operand of P.V; TMEM holds S, O and P of both tiles)
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    uint32_t pw[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        __nv_bfloat162 hh = __floats2bfloat162_rn(v[q4 * 32 + 2 * e], v[q4 * 32 + 2 * e + 1]);
                        pw[e] = *reinterpret_cast<uint32_t*>(&hh);
                    }
                    tmem_st16(tP + q4 * 16, pw);
                }
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&tail->pfull[t]);
                ++pc;
            }
            if (!ok) break;
            // the tile's output: O / l once its last P.V product is done
            if (!mbar_wait(&tail->oready[t], (pc - 1) & 1, abort_flag, P.status)) break;
            tc_fence_after();
            const float inv = row_ok ? 1.f / l : 0.f;
            __nv_bfloat16* orow = P.o + ((size_t)b * P.T + (row_ok ? row : 0)) * P.ld + (size_t)h * DH;
            #pragma unroll 1
            for (int c = 0; c < DH / 32; ++c) {
                uint32_t o[32];
                tmem_ld32(tO + c * 32, o);
                tmem_ld_wait();
                if (row_ok) {
#pragma unroll
                    for (int q8 = 0; q8 < 4; ++q8) {
                        __nv_bfloat162 hh[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            hh[e] = __floats2bfloat162_rn(__uint_as_float(o[q8 * 8 + 2 * e]) * inv,
                                                          __uint_as_float(o[q8 * 8 + 2 * e + 1]) * inv);
                        *reinterpret_cast<uint4*>(orow + c * 32 + q8 * 8) = *reinterpret_cast<uint4*>(hh);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tail->oempty[t]);
            // S_max: the raw max of the rows inside the sequence
            const float mw = warp_max_nan(row_ok ? m_raw : -INFINITY);
            if (lane == 0 && mw != -INFINITY)  // -inf: every row of this warp is past T
                merge_smax(mw, P.sqrt_d, P.s_max, P.s_bh, b, P.H, h, P.status);
        }
    }

    pdl_trigger();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_base, 512);
}

// ---------------------------------------------------------------------------
// MLA attention forward with the max logit taken along (K2's attention: the
// K2 review's MLA table).  Per head the logit is q^C.k^C over nope = 128
// plus q^R.k^R over rope = 64 with the k^R every head shares, d = 192; the
// values and the output have dv = 128.  The same kernel with NQK = 2 (no
// rope block) is the MHA forward at dh = 128.
//
// Same roles and item order as attn_kernel.  S_t = Q_t K_j^T runs over NQK
// 64-wide blocks: for MLA the two q^C blocks of the head against its k^C
// blocks and the q^R block against the shared k^R (loaded from its own
// tensor).  P_t goes to TMEM, over the first 64 columns of S_t (S0 | S1 |
// O0 | O1 fill the 512 columns), so shared memory holds only Q of two
// tiles, the K stages and two V stages (MLA: 96 + 48 + 64 KB; dh = 128:
// 64 + 2 x 32 + 64 KB), and no P tile is written to or read from it.  The
// MMA thread therefore issues S_t(j+1) only after O_t += P_t(j) V_j: the
// tensor pipe executes one thread's MMAs in issue order, so the product has
// read P before the next S overwrites it, and the softmax writes P_t(j) only
// after it has loaded S_t(j) and after the previous product (oready) has
// read P_t(j-1).
// ---------------------------------------------------------------------------
constexpr int kMlaQkBlocks = 3;  // q^C (2 blocks) and q^R (1 block) per head

// S_t = Q_t K^T over the NQK 64-wide blocks, the blocks in a rolled loop:
// the MMA warp runs on the smallest register share of the kernel
template <int NQK>
MC_D void issue_s_mla(uint32_t d_tmem, uint64_t qd, uint64_t kd, uint32_t idesc) {
#pragma unroll 1
    for (int c = 0; c < NQK; ++c) {
        const uint64_t boff = (uint64_t)((c * kAttnTile) >> 4);
#pragma unroll
        for (int k = 0; k < 4; ++k)
            umma_bf16(d_tmem, qd + boff + (uint64_t)(k * 2), kd + boff + (uint64_t)(k * 2), idesc, (c | k) != 0);
    }
}
constexpr int kMlaVBlocks = 2;   // dv = 128
// V gets two stages: V_{j+1} must land during block j (the next P.V waits
// on it first thing), while K_{j+1} is needed only after P_0(j) V_j has been
// issued and can load from the end of block j - 1 (measured: one V stage
// left the MMA thread waiting about 0.9 us for V every block).  MLA has room
// for one K stage, dh = 128 for two.
template <int NQK>
__host__ __device__ constexpr int mla_k_stages() { return NQK == kMlaQkBlocks ? 1 : 2; }
constexpr int kMlaVStages = 2;
static_assert((2 * kMlaQkBlocks + 1 * kMlaQkBlocks + kMlaVStages * kMlaVBlocks) * kAttnTile <= kAttnRing &&
                  (2 * 2 + 2 * 2 + kMlaVStages * kMlaVBlocks) * kAttnTile <= kAttnRing,
              "MLA shared memory");

template <int NQK>
__global__ void __launch_bounds__(kAttnThreads, 1) attn_mla_kernel(const __grid_constant__ AttnParams P) {
    constexpr int DV = 128;
    constexpr int kMlaKStages = mla_k_stages<NQK>();
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    AttnSmemTail* tail = reinterpret_cast<AttnSmemTail*>(smem);
    uint8_t* sQ = smem + 1024;                          // tile t: blocks NQK t ..
    uint8_t* sK = sQ + 2 * NQK * kAttnTile;            // stage s: NQK blocks (k^C, k^C[, k^R])
    uint8_t* sV = sK + kMlaKStages * NQK * kAttnTile;  // stage s: 2 blocks
    volatile int* abort_flag = &tail->abort_flag;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kAttnMaxStages; ++s) {
            mbar_init(&tail->kfull[s], 1);
            mbar_init(&tail->kempty[s], 1);
            mbar_init(&tail->vfull[s], 1);
            mbar_init(&tail->vempty[s], 1);
        }
        mbar_init(&tail->qfull, 1);
        mbar_init(&tail->qempty, 1);
        for (int t = 0; t < 2; ++t) {
            mbar_init(&tail->sfull[t], 1);
            mbar_init(&tail->sempty[t], 4);
            mbar_init(&tail->pfull[t], 4);
            mbar_init(&tail->oready[t], 1);
            mbar_init(&tail->oempty[t], 4);
        }
        mbar_init(&tail->drain, 1);
        tail->abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&P.tmQ);
        tma_prefetch_desc(&P.tmK);
        if (NQK == kMlaQkBlocks) tma_prefetch_desc(&P.tmKR);
        tma_prefetch_desc(&P.tmV);
    }
    if (warp == 1) {
        tmem_alloc(&tail->tmem_base, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = tail->tmem_base;  // S_t (and P_t) at 128 t, O_t at 256 + 128 t
    pdl_wait();

    if (warp < 4) {
    setmaxnreg_dec<kAttnRegsLow>();  // the dh = 64 split: P goes to TMEM here too
    if (warp == 0 || warp == 2) {
        // ---------------- TMA producers: Q and K (warp 0), V (warp 2) ----------------
        if (lane == 0) {
            const bool is_k = warp == 0;
            const int nst = is_k ? kMlaKStages : kMlaVStages;
            const int nblk = is_k ? NQK : kMlaVBlocks;
            uint64_t* full = is_k ? tail->kfull : tail->vfull;
            uint64_t* empty = is_k ? tail->kempty : tail->vempty;
            uint8_t* ring = is_k ? sK : sV;
            int stage = 0;
            uint32_t phase = 0;
            uint32_t issued[kAttnMaxStages] = {0, 0, 0, 0};
            uint32_t n = 0;
            bool ok = true;
            for (int r = 0, i = attn_round_item(0); i < P.total_items && ok; i = attn_round_item(++r), ++n) {
                int b, h, g, njb[2];
                attn_item(P, i, b, h, g, njb);
                if (is_k) {
                    if (!mbar_wait(&tail->qempty, (n & 1) ^ 1, abort_flag, P.status)) break;
                    mbar_arrive_expect_tx(&tail->qfull, 2 * NQK * kAttnTile);
                    for (int t = 0; t < 2; ++t)
                        for (int c = 0; c < NQK; ++c)
                            tma_load_3d(sQ + (t * NQK + c) * kAttnTile, &P.tmQ, &tail->qfull,
                                        h * (NQK * 64) + c * 64, (2 * g + t) * kAttnBlk, b);
                }
                const int nj = max(njb[0], njb[1]);
                for (int j = 0; j < nj; ++j) {
                    if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag, P.status)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&full[stage], nblk * kAttnTile);
                    uint8_t* dst = ring + stage * nblk * kAttnTile;
                    if (is_k) {
                        tma_load_3d(dst, &P.tmK, &full[stage], h * 128, j * kAttnBlk, b);
                        tma_load_3d(dst + kAttnTile, &P.tmK, &full[stage], h * 128 + 64, j * kAttnBlk, b);
                        if (NQK == kMlaQkBlocks)
                            tma_load_3d(dst + 2 * kAttnTile, &P.tmKR, &full[stage], P.kr_col, j * kAttnBlk, b);
                    } else {
                        tma_load_3d(dst, &P.tmV, &full[stage], h * DV, j * kAttnBlk, b);
                        tma_load_3d(dst + kAttnTile, &P.tmV, &full[stage], h * DV + 64, j * kAttnBlk, b);
                    }
                    ++issued[stage];
                    if (++stage == nst) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
            }
            volatile int never = 0;
            for (int s = 0; s < nst; ++s)
                if (issued[s]) mbar_wait(&full[s], (issued[s] - 1) & 1, &never, P.status);
            if (is_k && n) mbar_wait(&tail->qfull, (n - 1) & 1, &never, P.status);
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        const uint32_t idesc_s = idesc_f16kind(kAttnBlk, kAttnBlk, 0, 0);  // S = Q K^T, K-major K
        const uint32_t idesc_o = idesc_f16kind(kAttnBlk, DV, 1, 0);        // O += P V, MN-major V
        int ks = 0, vs = 0;
        uint32_t kph = 0, vph = 0;
        uint32_t pc[2] = {0, 0}, no[2] = {0, 0}, n = 0;
        bool ok = true;
        const uint64_t qdesc0 = sw128_desc(smem_u32(sQ), 16, 1024);
        const uint64_t kdesc0 = sw128_desc(smem_u32(sK), 16, 1024);
        const uint64_t vdesc0 = sw128_desc(smem_u32(sV), kAttnTile, 1024);
        const uint64_t qblk16 = (uint64_t)(NQK * kAttnTile) >> 4;  // one Q tile or one K stage
        const uint64_t vblk16 = (uint64_t)(kMlaVBlocks * kAttnTile) >> 4;   // one V stage
        auto issue_s_tile = [&](int t) {
            issue_s_mla<NQK>(tmem_base + t * kAttnBlk, qdesc0 + (uint64_t)t * qblk16, kdesc0 + (uint64_t)ks * qblk16,
                        idesc_s);
            umma_commit(&tail->sfull[t]);
        };
        for (int r = 0, i = attn_round_item(0); i < P.total_items && ok; i = attn_round_item(++r), ++n) {
            int b, h, g, njb[2];
            attn_item(P, i, b, h, g, njb);
            const int nj = max(njb[0], njb[1]);
            if (!mbar_wait(&tail->qfull, n & 1, abort_flag, P.status)) break;
            // S_t(0) of both tiles
            if (!mbar_wait(&tail->kfull[ks], kph, abort_flag, P.status)) break;
            tc_fence_after();
            if (lane == 0) {
#pragma unroll
                for (int t = 0; t < 2; ++t)
                    if (njb[t] > 0) issue_s_tile(t);
                umma_commit(&tail->kempty[ks]);
                if (nj == 1) umma_commit(&tail->qempty);
            }
            __syncwarp();
            if (++ks == kMlaKStages) {
                ks = 0;
                kph ^= 1;
            }
            for (int j = 0; j < nj && ok; ++j) {
                // O_t += P_t(j) V_j, then S_t(j + 1) into the columns P_t(j) occupied
                if (!mbar_wait(&tail->vfull[vs], vph, abort_flag, P.status)) {
                    ok = false;
                    break;
                }
                const bool next_k = j + 1 < nj;
                bool have_k = false;  // K_{j+1} landed: waited for just before its first use
#pragma unroll
                for (int t = 0; t < 2; ++t) {
                    if (!ok || j >= njb[t]) continue;
                    if (j == 0 && !mbar_wait(&tail->oempty[t], (no[t] & 1) ^ 1, abort_flag, P.status)) ok = false;
                    if (ok && !mbar_wait(&tail->pfull[t], pc[t] & 1, abort_flag, P.status)) ok = false;
                    if (!ok) continue;
                    tc_fence_after();
                    if (lane == 0) {
                        issue_pv_tmem_a(tmem_base + 256 + t * DV, tmem_base + t * kAttnBlk,
                                        vdesc0 + (uint64_t)vs * vblk16, idesc_o, j != 0);
                        umma_commit(&tail->oready[t]);
                    }
                    __syncwarp();
                    if (j + 1 < njb[t]) {
                        if (!have_k) {
                            if (!mbar_wait(&tail->kfull[ks], kph, abort_flag, P.status)) {
                                ok = false;
                                continue;
                            }
                            tc_fence_after();
                            have_k = true;
                        }
                        if (lane == 0) issue_s_tile(t);
                        __syncwarp();
                    }
                    ++pc[t];
                    if (j == njb[t] - 1) ++no[t];
                }
                if (!ok) break;
                if (lane == 0) {
                    umma_commit(&tail->vempty[vs]);  // V_j consumed by both tiles
                    if (next_k) {
                        umma_commit(&tail->kempty[ks]);                // K_{j+1} consumed
                        if (j + 1 == nj - 1) umma_commit(&tail->qempty);  // the item's last use of Q
                    }
                }
                __syncwarp();
                if (++vs == kMlaVStages) {
                    vs = 0;
                    vph ^= 1;
                }
                if (next_k && ++ks == kMlaKStages) {
                    ks = 0;
                    kph ^= 1;
                }
            }
        }
        if (lane == 0) umma_commit(&tail->drain);
        __syncwarp();
        volatile int never = 0;
        mbar_wait(&tail->drain, 0, &never, P.status);
    }
    } else {
        setmaxnreg_inc<kAttnRegsHigh>();
        // ---------------- softmax and output: tile t = warpgroup - 1 ----------------
        const int t = warp >= 8 ? 1 : 0;
        const int quarter = warp & 3;
        const int lr = quarter * 32 + lane;
        const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
        const uint32_t tS = tmem_base + lane_base + t * kAttnBlk;  // S_t, and P_t over its first 64 columns
        const uint32_t tO = tmem_base + lane_base + 256 + t * DV;
        uint32_t sc = 0, pc = 0;
        bool ok = true;
        for (int r = 0, i = attn_round_item(0); i < P.total_items && ok; i = attn_round_item(++r)) {
            int b, h, g, njb[2];
            attn_item(P, i, b, h, g, njb);
            const int nj = njb[t];
            if (nj == 0) continue;
            const int it = 2 * g + t;
            const int row = it * kAttnBlk + lr;
            const bool row_ok = row < P.T;
            float m = -INFINITY, l = 0.f, m_raw = -INFINITY;
            for (int j = 0; j < nj && ok; ++j) {
                if (!mbar_wait(&tail->sfull[t], sc & 1, abort_flag, P.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                float v[kAttnBlk];
                uint32_t* vu = reinterpret_cast<uint32_t*>(v);
#pragma unroll
                for (int c = 0; c < kAttnBlk / 32; ++c) tmem_ld32(tS + c * 32, vu + c * 32);
                tmem_ld_wait();
                ++sc;
                const int key0 = j * kAttnBlk;
                const bool full = (it + 1) * kAttnBlk <= P.T && key0 + kAttnBlk <= P.T &&
                                  (!P.causal || key0 + kAttnBlk - 1 <= it * kAttnBlk);
                if (!full) {
                    const int lim = !row_ok ? 0 : (P.causal ? min(row + 1, P.T) : P.T);
#pragma unroll
                    for (int e = 0; e < kAttnBlk; ++e)
                        if (key0 + e >= lim) v[e] = -INFINITY;
                }
                float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                for (int e = 0; e < kAttnBlk; e += 8)
#pragma unroll
                    for (int c = 0; c < 4; ++c) m4[c] = max3_nan(m4[c], v[e + 2 * c], v[e + 2 * c + 1]);
                const float mb = max_nan(max_nan(m4[0], m4[1]), max_nan(m4[2], m4[3]));
                m_raw = max_nan(m_raw, mb);
                const float mx = mb * P.scale_log2;
                const float m_new = !row_ok ? 0.f : (mx > m + 8.f || m == -INFINITY) ? fmaxf(m, mx) : m;
                const float alpha = row_ok && m_new != m ? ex2_approx(m - m_new) : 1.f;
                // pairs of logits through the packed fp32 FMA and add of
                // sm_100+; logit e goes to partial sum e mod 8
                const float2 sc2 = make_float2(P.scale_log2, P.scale_log2), nm2 = make_float2(-m_new, -m_new);
                float2 ls[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                                make_float2(0.f, 0.f)};
#pragma unroll
                for (int e = 0; e < kAttnBlk; e += 2) {
                    const float2 x = __ffma2_rn(make_float2(v[e], v[e + 1]), sc2, nm2);
                    const float p0 = row_ok ? ex2_approx(x.x) : 0.f, p1 = row_ok ? ex2_approx(x.y) : 0.f;
                    v[e] = p0;
                    v[e + 1] = p1;
                    ls[(e >> 1) & 3] = __fadd2_rn(ls[(e >> 1) & 3], make_float2(p0, p1));
                }
                const float lsum = ((ls[0].x + ls[0].y) + (ls[1].x + ls[1].y)) + ((ls[2].x + ls[2].y) + (ls[3].x + ls[3].y));
                l = __fmaf_rn(l, alpha, lsum);
                m = m_new;
                if (j >= 1) {
                    // O_t is free (and P_t(j-1) read) once P_{j-1} V_{j-1} is done
                    if (!mbar_wait(&tail->oready[t], (pc - 1) & 1, abort_flag, P.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    if (__any_sync(0xFFFFFFFFu, alpha != 1.f)) {
                        #pragma unroll 1
                        for (int c = 0; c < DV / 32; ++c) {
                            uint32_t o[32];
                            tmem_ld32(tO + c * 32, o);
                            tmem_ld_wait();
#pragma unroll
                            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                            tmem_st32(tO + c * 32, o);
                        }
                    }
                }
                // P_t(j) as bf16 pairs over S_t's first 64 columns
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    uint32_t pw[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        __nv_bfloat162 hh = __floats2bfloat162_rn(v[q4 * 32 + 2 * e], v[q4 * 32 + 2 * e + 1]);
                        pw[e] = *reinterpret_cast<uint32_t*>(&hh);
                    }
                    tmem_st16(tS + q4 * 16, pw);
                }
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&tail->pfull[t]);
                ++pc;
            }
            if (!ok) break;
            if (!mbar_wait(&tail->oready[t], (pc - 1) & 1, abort_flag, P.status)) break;
            tc_fence_after();
            const float inv = row_ok ? 1.f / l : 0.f;
            __nv_bfloat16* orow = P.o + ((size_t)b * P.T + (row_ok ? row : 0)) * P.ld + (size_t)h * DV;
            #pragma unroll 1
            for (int c = 0; c < DV / 32; ++c) {
                uint32_t o[32];
                tmem_ld32(tO + c * 32, o);
                tmem_ld_wait();
                if (row_ok) {
#pragma unroll
                    for (int q8 = 0; q8 < 4; ++q8) {
                        __nv_bfloat162 hh[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            hh[e] = __floats2bfloat162_rn(__uint_as_float(o[q8 * 8 + 2 * e]) * inv,
                                                          __uint_as_float(o[q8 * 8 + 2 * e + 1]) * inv);
                        *reinterpret_cast<uint4*>(orow + c * 32 + q8 * 8) = *reinterpret_cast<uint4*>(hh);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tail->oempty[t]);
            const float mw = warp_max_nan(row_ok ? m_raw : -INFINITY);
            if (lane == 0 && mw != -INFINITY)  // -inf: every row of this warp is past T
                merge_smax(mw, P.sqrt_d, P.s_max, P.s_bh, b, P.H, h, P.status);
        }
    }

    pdl_trigger();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_base, 512);
}

// Items per band of the MHA forward: eight rounds.  With few (sequence,
// head) pairs the causal tail is the limit, and the heavy-first order within
// a band only balances it when the band spans many rounds: [2, 8192, 16
// heads] causal ran 0.485 ms at dh = 128 and 0.414 ms at dh = 64 with one
// band of all 32 pairs, against 0.609 and 0.525 ms with two rounds per band.
static int attn_band_items(int grid) { return 8 * grid; }

// The P-in-TMEM kernel: MLA (d = 192 over q^C, k^C and the shared k^R) or,
// with NQK = 2, MHA at dh = 128.
template <int NQK>
static cudaError_t launch_attn_tmem_p(const AttnArgs& a, cudaStream_t stream) {
    AttnParams P;
    memset(&P, 0, sizeof(P));
    constexpr int d = NQK * 64;
    const uint64_t q_ld = (uint64_t)a.H * d, kv_ld = (uint64_t)a.H * 128;
    if (!make_tmap_3d(&P.tmQ, a.q, q_ld, a.T, a.B, q_ld, q_ld * a.T, 64, kAttnBlk, 0)) return cudaErrorInvalidValue;
    if (!make_tmap_3d(&P.tmK, a.k, kv_ld, a.T, a.B, kv_ld, kv_ld * a.T, 64, kAttnBlk, 0)) return cudaErrorInvalidValue;
    if (!make_tmap_3d(&P.tmV, a.v, kv_ld, a.T, a.B, kv_ld, kv_ld * a.T, 64, kAttnBlk, 0)) return cudaErrorInvalidValue;
    if (NQK == kMlaQkBlocks) {
        if (!make_tmap_3d(&P.tmKR, a.kr, (uint64_t)a.kr_ld, a.T, a.B, (uint64_t)a.kr_ld, (uint64_t)a.kr_ld * a.T, 64,
                          kAttnBlk, 0))
            return cudaErrorInvalidValue;
        P.kr_col = a.kr_col;
    } else {
        P.tmKR = P.tmK;  // not read
    }
    P.B = a.B;
    P.T = a.T;
    P.H = a.H;
    P.dh = d;
    P.causal = a.causal;
    P.n_it = (a.T + kAttnBlk - 1) / kAttnBlk;
    P.n_pair = (P.n_it + 1) / 2;
    P.total_items = a.B * a.H * P.n_pair;
    P.o = reinterpret_cast<__nv_bfloat16*>(a.o);
    P.ld = (long long)kv_ld;
    P.scale_log2 = (float)(1.4426950408889634 / sqrt((double)d));
    P.sqrt_d = sqrtf((float)d);
    P.s_max = a.s_max;
    P.s_bh = a.s_bh;
    P.status = device_status_ptr();
    P.kst = mla_k_stages<NQK>();
    P.vst = kMlaVStages;
    static bool attr_set[64] = {false};
    int dev = current_device();
    if (dev < 0) return cudaErrorInvalidDevice;
    if (dev < 64 && !attr_set[dev]) {
        cudaError_t e =
            cudaFuncSetAttribute(attn_mla_kernel<NQK>, cudaFuncAttributeMaxDynamicSharedMemorySize, kAttnSmem);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    int grid = num_sms();
    if (grid > P.total_items) grid = P.total_items;
    // items per band: MLA a quarter of a round (its K and V, with a 16 KB
    // row stride at K2's 64 heads, were re-read from DRAM three times over
    // with two rounds: 2.28 ms with a quarter, 2.35 with a half, 2.55 with two
    // at [2, 8192, 64 heads]); MHA eight rounds (attn_band_items)
    const int band_items = NQK == kMlaQkBlocks ? grid / 4 : attn_band_items(grid);
    P.band = std::max(1, std::min(a.B * a.H, (band_items + P.n_pair - 1) / P.n_pair));
    TraceScope ts(NQK == kMlaQkBlocks ? "attn_mla" : "attn", stream);
    return launch_pdl(attn_mla_kernel<NQK>, dim3(grid), dim3(kAttnThreads), kAttnSmem, stream, P);
}

cudaError_t launch_attn(const AttnArgs& a, cudaStream_t stream) {
    if (a.mla) return launch_attn_tmem_p<kMlaQkBlocks>(a, stream);
    if (a.dh == 128) return launch_attn_tmem_p<2>(a, stream);
    AttnParams P;
    memset(&P, 0, sizeof(P));
    if (a.dh != 64) return cudaErrorInvalidValue;
    const uint64_t ld = (uint64_t)a.H * a.dh;
    if (!make_tmap_3d(&P.tmQ, a.q, ld, a.T, a.B, ld, ld * a.T, 64, kAttnBlk, 0)) return cudaErrorInvalidValue;
    if (!make_tmap_3d(&P.tmK, a.k, ld, a.T, a.B, ld, ld * a.T, 64, kAttnBlk, 0)) return cudaErrorInvalidValue;
    if (!make_tmap_3d(&P.tmV, a.v, ld, a.T, a.B, ld, ld * a.T, 64, kAttnBlk, 0)) return cudaErrorInvalidValue;
    P.B = a.B;
    P.T = a.T;
    P.H = a.H;
    P.dh = a.dh;
    P.causal = a.causal;
    P.n_it = (a.T + kAttnBlk - 1) / kAttnBlk;
    P.n_pair = (P.n_it + 1) / 2;
    P.total_items = a.B * a.H * P.n_pair;
    P.o = reinterpret_cast<__nv_bfloat16*>(a.o);
    P.ld = (long long)ld;
    P.scale_log2 = (float)(1.4426950408889634 / sqrt((double)a.dh));
    P.sqrt_d = sqrtf((float)a.dh);
    P.s_max = a.s_max;
    P.s_bh = a.s_bh;
    P.status = device_status_ptr();
    // after Q of two tiles: K and V rings of 4 + 4 one-block stages
    P.kst = 4;
    P.vst = 4;
    static_assert((2 + 4 + 4) * kAttnTile <= kAttnRing, "attention shared memory");
    static bool attr_set[64] = {false};
    int dev = current_device();
    if (dev < 0) return cudaErrorInvalidDevice;
    if (dev < 64 && !attr_set[dev]) {
        cudaError_t e = cudaFuncSetAttribute(attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kAttnSmem);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    int grid = num_sms();
    if (grid > P.total_items) grid = P.total_items;
    P.band = std::max(1, std::min(a.B * a.H, (attn_band_items(grid) + P.n_pair - 1) / P.n_pair));
    TraceScope ts("attn", stream);
    return launch_pdl(attn_kernel, dim3(grid), dim3(kAttnThreads), kAttnSmem, stream, P);
}

}  // namespace mc
