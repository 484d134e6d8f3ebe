// Attention forward of an MHA layer with the max logit taken along: the
// softmax inputs s_ij = q_i . k_j are computed anyway, so S_max^h of the
// MuonClip step ("Kimi K2" section 2.1 and the K2 notes: the clip uses the
// max logit of this step and leaves the forward unchanged) costs one max per
// logit on top of O = softmax(Q K^T / sqrt(dh)) V.
//
// Work item = (sequence b, head h, 128-query tile); one persistent CTA per
// SM; items in bands of (b, h) pairs dealt in snake-ordered rounds (as in
// the scan).  Per 128-key block j of an item:
//   warp 0      TMA: the item's Q tile once, the K_j and V_j tiles (128 keys
//               x dh) into a ring of stages
//   warp 1      tcgen05.mma S_j = Q K_j^T into one of two 128 x 128 fp32
//               TMEM tiles; once P_j is ready, O += P_j V_j into the
//               128 x dh fp32 TMEM accumulator (P from shared memory, V
//               MN-major as stored)
//   warps 2..5  one query row per lane: S_j from TMEM, the raw row max (for
//               S_max), the running softmax max m and sum l, O rescaled by
//               2^(m_old - m_new) in TMEM when m grows, P_j = 2^(s - m) as
//               bf16 into a swizzled shared tile; at the end of the item
//               O / l as bf16 and one atomicMax per warp on the monotonic key
//               of (b, h)
// The last CTA turns the keys into S_max (key / sqrt(dh)), like the scan.
#include "common.cuh"
#include "internal.h"

namespace mc {

constexpr int kAttnThreads = 192;
constexpr int kAttnBlk = 128;          // queries per item, keys per key block
constexpr int kAttnMaxStages = 4;
constexpr int kAttnTile = 16384;       // 128 rows x 64 bf16 (one 128-byte-swizzled block)
constexpr int kAttnRing = 224 * 1024;  // Q + two P tiles + K/V stages
constexpr int kAttnSmem = 1024 + 1024 + kAttnRing;

struct AttnParams {
    CUtensorMap tmQ, tmK, tmV;  // {H*dh, T, B} bf16, box {64, 128}
    int B, T, H, dh, causal;
    int n_it, total_items, band, stages;
    __nv_bfloat16* o;
    long long ld;               // H * dh: row stride of q, k, v and o
    float scale_log2;           // log2(e) / sqrt(dh)
    unsigned* keys;             // [B*H] monotonic keys of the raw max, then a done counter
    unsigned* done;
    float sqrt_d;
    int accumulate;
    float* s_max;
    float* s_bh;
    unsigned* status;
};

struct AttnSmemTail {
    uint64_t kvfull[kAttnMaxStages], kvempty[kAttnMaxStages];
    uint64_t qfull, qempty;
    uint64_t sfull[2], sempty[2];
    uint64_t pfull[2];
    uint64_t oready;  // one phase per P.V product
    uint64_t oempty;  // the item's output has been read from TMEM
    uint64_t drain;
    uint32_t tmem_base;
    int abort_flag;
    int last_cta;
};

// 2^x with the hardware approximation (relative error about 2^-22, far below
// the bf16 rounding of the softmax weights; tiny results flush to zero)
MC_D float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

MC_D void attn_item(const AttnParams& P, int i, int& b, int& h, int& it, int& njb) {
    const int BH = P.B * P.H;
    const int per_band = P.band * P.n_it;
    const int band = i / per_band;
    const int w = i - band * per_band;
    const int pairs = min(P.band, BH - band * P.band);
    const int grp = w / pairs;
    const int bh = band * P.band + (w - grp * pairs);
    it = P.causal ? (P.n_it - 1 - grp) : grp;  // heaviest causal tiles first
    b = bh / P.H;
    h = bh - b * P.H;
    const int row_end = min(P.T, (it + 1) * kAttnBlk);
    njb = P.causal ? (row_end - 1) / kAttnBlk + 1 : (P.T + kAttnBlk - 1) / kAttnBlk;
}

MC_D int attn_round_item(int r) {
    const int c = (r & 1) ? (int)(gridDim.x - 1 - blockIdx.x) : (int)blockIdx.x;
    return r * (int)gridDim.x + c;
}

__global__ void __launch_bounds__(kAttnThreads, 1) attn_kernel(const __grid_constant__ AttnParams P) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    static_assert(sizeof(AttnSmemTail) <= 1024, "tail");
    AttnSmemTail* tail = reinterpret_cast<AttnSmemTail*>(smem);
    const int nc = P.dh / 64;                 // 64-column blocks per row of q, k, v
    const int nst = P.stages;
    uint8_t* sQ = smem + 1024;                // nc blocks
    uint8_t* sP = sQ + nc * kAttnTile;        // two P tiles of 2 blocks (128 keys)
    uint8_t* sKV = sP + 4 * kAttnTile;        // stage s: K at sKV + s * 2nc blocks, V after it
    volatile int* abort_flag = &tail->abort_flag;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t kv_bytes = (uint32_t)(2 * nc * kAttnTile);

    if (threadIdx.x == 0) {
        for (int s = 0; s < nst; ++s) {
            mbar_init(&tail->kvfull[s], 1);
            mbar_init(&tail->kvempty[s], 1);
        }
        mbar_init(&tail->qfull, 1);
        mbar_init(&tail->qempty, 1);
        for (int a = 0; a < 2; ++a) {
            mbar_init(&tail->sfull[a], 1);
            mbar_init(&tail->sempty[a], 4);
            mbar_init(&tail->pfull[a], 4);
        }
        mbar_init(&tail->oready, 1);
        mbar_init(&tail->oempty, 4);
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
    const uint32_t tmem_base = tail->tmem_base;
    const uint32_t tO = tmem_base + 256;      // S tiles at columns 0 and 128, O after them
    pdl_wait();

    if (warp == 0) {
        // ---------------- TMA producer ----------------
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t issued[kAttnMaxStages] = {0, 0, 0, 0};
            uint32_t n = 0;
            bool ok = true;
            for (int r = 0, i = attn_round_item(0); i < P.total_items && ok; i = attn_round_item(++r), ++n) {
                int b, h, it, njb;
                attn_item(P, i, b, h, it, njb);
                if (!mbar_wait(&tail->qempty, (n & 1) ^ 1, abort_flag, P.status)) break;
                mbar_arrive_expect_tx(&tail->qfull, (uint32_t)(nc * kAttnTile));
                for (int c = 0; c < nc; ++c)
                    tma_load_3d(sQ + c * kAttnTile, &P.tmQ, &tail->qfull, h * P.dh + c * 64, it * kAttnBlk, b);
                for (int j = 0; j < njb; ++j) {
                    if (!mbar_wait(&tail->kvempty[stage], phase ^ 1, abort_flag, P.status)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&tail->kvfull[stage], kv_bytes);
                    uint8_t* sk = sKV + stage * 2 * nc * kAttnTile;
                    for (int c = 0; c < nc; ++c) {
                        tma_load_3d(sk + c * kAttnTile, &P.tmK, &tail->kvfull[stage], h * P.dh + c * 64,
                                    j * kAttnBlk, b);
                        tma_load_3d(sk + (nc + c) * kAttnTile, &P.tmV, &tail->kvfull[stage], h * P.dh + c * 64,
                                    j * kAttnBlk, b);
                    }
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
                if (issued[s]) mbar_wait(&tail->kvfull[s], (issued[s] - 1) & 1, &never, P.status);
            if (n) mbar_wait(&tail->qfull, (n - 1) & 1, &never, P.status);
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        const uint32_t idesc_s = idesc_f16kind(kAttnBlk, kAttnBlk, 0, 0);  // S = Q K^T, K-major K
        const uint32_t idesc_o = idesc_f16kind(kAttnBlk, P.dh, 1, 0);      // O += P V, MN-major V
        int stage = 0;
        uint32_t phase = 0;
        uint32_t sc = 0, pc = 0, n = 0;  // S tiles, P.V products, items
        bool ok = true;
        // O += P_j V_j for the block in ring stage st; the first of an item
        // overwrites O once the previous item's output has been read
        auto pv = [&](int j, int st) {
            if (j == 0 && !mbar_wait(&tail->oempty, (n & 1) ^ 1, abort_flag, P.status)) return false;
            if (!mbar_wait(&tail->pfull[pc & 1], (pc >> 1) & 1, abort_flag, P.status)) return false;
            tc_fence_after();
            if (lane == 0) {
                const uint32_t p0 = smem_u32(sP + (pc & 1) * 2 * kAttnTile);
                const uint32_t v0 = smem_u32(sKV + st * 2 * nc * kAttnTile + nc * kAttnTile);
#pragma unroll
                for (int k = 0; k < kAttnBlk / 16; ++k) {
                    const uint64_t ad = sw128_desc(p0 + (k >> 2) * kAttnTile + (k & 3) * 32, 16, 1024);
                    const uint64_t bd = sw128_desc(v0 + k * 2048, kAttnTile, 1024);
                    umma_bf16(tO, ad, bd, idesc_o, (j | k) != 0);
                }
                umma_commit(&tail->oready);
                umma_commit(&tail->kvempty[st]);  // K_j and V_j are both consumed now
            }
            __syncwarp();
            ++pc;
            return true;
        };
        for (int r = 0, i = attn_round_item(0); i < P.total_items && ok; i = attn_round_item(++r), ++n) {
            int b, h, it, njb;
            attn_item(P, i, b, h, it, njb);
            if (!mbar_wait(&tail->qfull, n & 1, abort_flag, P.status)) break;
            tc_fence_after();
            const uint32_t q0 = smem_u32(sQ);
            int prev_stage = -1;
            for (int j = 0; j < njb && ok; ++j) {
                // S_j = Q K_j^T
                if (!mbar_wait(&tail->kvfull[stage], phase, abort_flag, P.status) ||
                    !mbar_wait(&tail->sempty[sc & 1], ((sc >> 1) & 1) ^ 1, abort_flag, P.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (lane == 0) {
                    const uint32_t k0 = smem_u32(sKV + stage * 2 * nc * kAttnTile);
                    const uint32_t ts = tmem_base + (sc & 1) * kAttnBlk;
                    for (int k = 0; k < P.dh / 16; ++k) {
                        const uint32_t off = (k >> 2) * kAttnTile + (k & 3) * 32;
                        umma_bf16(ts, sw128_desc(q0 + off, 16, 1024), sw128_desc(k0 + off, 16, 1024), idesc_s,
                                  k != 0);
                    }
                    umma_commit(&tail->sfull[sc & 1]);
                    if (j == njb - 1) umma_commit(&tail->qempty);  // the item's last use of Q
                }
                __syncwarp();
                ++sc;
                const int cur = stage;
                if (++stage == nst) {
                    stage = 0;
                    phase ^= 1;
                }
                // O += P_{j-1} V_{j-1} while the softmax works on S_j
                if (j >= 1 && !pv(j - 1, prev_stage)) {
                    ok = false;
                    break;
                }
                prev_stage = cur;
            }
            if (!ok) break;
            if (!pv(njb - 1, prev_stage)) break;
        }
        if (lane == 0) umma_commit(&tail->drain);
        __syncwarp();
        volatile int never = 0;
        mbar_wait(&tail->drain, 0, &never, P.status);
    } else {
        // ---------------- softmax and output (warps 2..5) ----------------
        const int quarter = warp & 3;  // TMEM lanes 32 q .. 32 q + 31
        const int lr = quarter * 32 + lane;  // row of the item's tile
        const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
        uint32_t sc = 0, pc = 0, n = 0;
        bool ok = true;
        for (int r = 0, i = attn_round_item(0); i < P.total_items && ok; i = attn_round_item(++r), ++n) {
            int b, h, it, njb;
            attn_item(P, i, b, h, it, njb);
            const int row = it * kAttnBlk + lr;
            const bool row_ok = row < P.T;
            float m = -INFINITY, l = 0.f, m_raw = -INFINITY;
            for (int j = 0; j < njb && ok; ++j) {
                if (!mbar_wait(&tail->sfull[sc & 1], (sc >> 1) & 1, abort_flag, P.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                float v[kAttnBlk];
                uint32_t* vu = reinterpret_cast<uint32_t*>(v);
                const uint32_t ts = tmem_base + lane_base + (sc & 1) * kAttnBlk;
#pragma unroll
                for (int c = 0; c < kAttnBlk / 32; ++c) tmem_ld32(ts + c * 32, vu + c * 32);
                tmem_ld_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&tail->sempty[sc & 1]);
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
                float ls[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};  // eight partial sums
#pragma unroll
                for (int e = 0; e < kAttnBlk; ++e) {
                    const float p = row_ok ? ex2_approx(__fmaf_rn(v[e], P.scale_log2, -m_new)) : 0.f;
                    v[e] = p;
                    ls[e & 7] += p;
                }
                const float lsum = ((ls[0] + ls[1]) + (ls[2] + ls[3])) + ((ls[4] + ls[5]) + (ls[6] + ls[7]));
                l = __fmaf_rn(l, alpha, lsum);
                m = m_new;
                if (j >= 1) {
                    // O and P tile (pc & 1) are free once P_{j-1} V_{j-1} is done
                    if (!mbar_wait(&tail->oready, (pc - 1) & 1, abort_flag, P.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    if (__any_sync(0xFFFFFFFFu, alpha != 1.f)) {
                        for (int c = 0; c < P.dh / 32; ++c) {
                            uint32_t o[32];
                            tmem_ld32(tO + lane_base + c * 32, o);
                            tmem_ld_wait();
#pragma unroll
                            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                            tmem_st32(tO + lane_base + c * 32, o);
                        }
                        tmem_st_wait();
                    }
                }
                // P_j as bf16, 128-byte swizzled K-major rows (two 64-key blocks)
                uint8_t* pt = sP + (pc & 1) * 2 * kAttnTile;
#pragma unroll
                for (int cc = 0; cc < kAttnBlk / 8; ++cc) {
                    __nv_bfloat162 hh[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) hh[e] = __floats2bfloat162_rn(v[cc * 8 + 2 * e], v[cc * 8 + 2 * e + 1]);
                    *reinterpret_cast<uint4*>(pt + (cc >> 3) * kAttnTile + lr * 128 + (((cc & 7) ^ (lr & 7)) << 4)) =
                        *reinterpret_cast<uint4*>(hh);
                }
                fence_proxy_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&tail->pfull[pc & 1]);
                ++pc;
            }
            if (!ok) break;
            // the item's output: O / l once the last P.V product is done
            if (!mbar_wait(&tail->oready, (pc - 1) & 1, abort_flag, P.status)) break;
            tc_fence_after();
            const float inv = row_ok ? 1.f / l : 0.f;
            __nv_bfloat16* orow = P.o + ((size_t)b * P.T + (row_ok ? row : 0)) * P.ld + (size_t)h * P.dh;
            for (int c = 0; c < P.dh / 32; ++c) {
                uint32_t o[32];
                tmem_ld32(tO + lane_base + c * 32, o);
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
            if (lane == 0) mbar_arrive(&tail->oempty);
            // S_max: the raw max of the rows inside the sequence
            const float mw = warp_max_nan(row_ok ? m_raw : -INFINITY);
            if (lane == 0 && mw != -INFINITY) atomicMax(&P.keys[b * P.H + h], float_key(mw));
        }
    }

    pdl_trigger();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_base, 512);
    // the last CTA to finish turns the keys into S_max
    if (threadIdx.x == 0) {
        __threadfence();
        const unsigned old = atomicAdd(P.done, 1u);
        tail->last_cta = old == gridDim.x - 1;
    }
    __syncthreads();
    if (tail->last_cta) {
        __threadfence();
        for (int h = threadIdx.x; h < P.H; h += blockDim.x)
            finalize_head(P.keys, P.B, P.H, h, P.sqrt_d, P.accumulate, P.s_max, P.s_bh, P.status);
    }
}

cudaError_t launch_attn(const AttnArgs& a, cudaStream_t stream) {
    AttnParams P;
    memset(&P, 0, sizeof(P));
    if (a.dh != 64 && a.dh != 128) return cudaErrorInvalidValue;
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
    P.total_items = a.B * a.H * P.n_it;
    P.o = reinterpret_cast<__nv_bfloat16*>(a.o);
    P.ld = (long long)ld;
    P.scale_log2 = (float)(1.4426950408889634 / sqrt((double)a.dh));
    P.keys = a.keys;
    P.done = a.keys + (size_t)a.B * a.H;
    P.sqrt_d = sqrtf((float)a.dh);
    P.accumulate = a.accumulate;
    P.s_max = a.s_max;
    P.s_bh = a.s_bh;
    P.status = device_status_ptr();
    const int nc = a.dh / 64;
    // stages of K + V tiles after Q and two P tiles (4 at dh = 64, 2 at 128)
    P.stages = std::min(kAttnMaxStages, (kAttnRing - (nc + 4) * kAttnTile) / (2 * nc * kAttnTile));
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
    P.band = std::max(1, std::min(a.B * a.H, (2 * grid + P.n_it - 1) / P.n_it));
    TraceScope ts("attn", stream);
    return launch_pdl(attn_kernel, dim3(grid), dim3(kAttnThreads), kAttnSmem, stream, P);
}

}  // namespace mc
