// scan.cu -- per-head max-logit scan on tcgen05 tensor cores (sm_103a).
//
// S_max^h = max_{X,i,j} Q_i^h K_j^h / sqrt(d) ("Kimi K2: 1T MoE, MuonClip and
// Agentic training system", S_max equation; Kimi K2 section 2.1), computed
// tile by tile without ever storing the T x T logits.
//
// Q and K arrive in fp16 (the projections round their fp32 accumulators
// once to fp16: 11 significant bits keep S_max within 1e-3 of the exact
// value, where bf16's 8 do not); the MMAs are kind::f16 with F16 operands.
//
// Work item = (sequence b, head h, 128-query tile).  One persistent CTA per
// SM; items are dealt round-robin, heaviest causal rows first.
//   warp 0      TMA: the item's Q tile (128 x d, d/64 blocks) once, then the
//               K tiles (256 keys x 64) of every key tile into a ring of up to
//               6 stages
//   warp 1      tcgen05.mma Q K^T into one of two 128 x 256 fp32 TMEM tiles
//   warps 2..5  tcgen05.ld -> running row max (max.NaN, 4 chains) with the
//               causal / sequence-end mask only on edge tiles; at the end of
//               the item a warp max, and per warp S = max / sqrt(d)
//               max-merged into S_max[h] (and S_max[b, h]) by one integer
//               atomic each: the outputs need no pass after the scan
// MLA items accumulate d = nope + rope = 192 as three K blocks: two q^C.k^C
// blocks from the per-head k^C storage and one q^R.k^R block from the
// shared k^R storage, all into the same TMEM tile.
#include "common.cuh"
#include "internal.h"

namespace mc {

// Shared memory: a 1 KB block with the barriers, two Q buffers of nkb 16 KB
// blocks each, then as many 32 KB K stages as fit in 224 KB: 6 at d = 64
// (more K tiles in flight), 4 at d = 192.
constexpr int kScanMaxStages = 6;
constexpr int kScanQBlocks = 3;                  // d up to 192 per Q buffer
constexpr int kScanRing = 224 * 1024;            // Q buffers + K stages
constexpr int kQBlockBytes = kBM * kBK * 2;      // 16 KB
constexpr int kKStageBytes = kBN * kBK * 2;      // 32 KB
constexpr int kScanThreads = 192;
constexpr int kScanSmem = 1024 + 1024 + kScanRing;

struct ScanParams {
    CUtensorMap tmQ;   // {q_ld, T, B}, box {64, 128}
    CUtensorMap tmK;   // {k_ld, T, B}, box {64, 256}
    CUtensorMap tmKR;  // {kr_ld, T, B}, box {64, 256} (MLA k^R)
    int B, T, H, causal;
    int q_head_stride, k_head_stride, nkb_main, nkb_rope, kr_col;
    int n_it, total_items;
    int band;    // (sequence, head) pairs per band of the item order
    int stages;  // K stages in the ring
    float sqrt_d;
    float* s_max;  // filled with 0xFFFFFFFF, or holding the maxima to merge into
    float* s_bh;
    unsigned* status;
};

struct ScanSmemTail {
    uint64_t kfull[kScanMaxStages];
    uint64_t kempty[kScanMaxStages];
    uint64_t qfull[2], qempty[2];
    uint64_t tfull[2];
    uint64_t tempty[2];
    uint64_t drain;
    uint32_t tmem_base;
    int abort_flag;
};


// Item order: bands of P.band (sequence, head) pairs; within a band the
// query tiles go heaviest causal tile first, pairs minor.  The items running
// at one time then share the K panels of a few pairs (which stay in L2)
// instead of touching one panel per CTA.
MC_D void decode_item(const ScanParams& P, int i, int& b, int& h, int& it, int& njt) {
    const int BH = P.B * P.H;
    const int per_band = P.band * P.n_it;
    const int band = i / per_band;
    const int w = i - band * per_band;
    const int pairs = min(P.band, BH - band * P.band);  // the last band may be short
    const int grp = w / pairs;
    const int bh = band * P.band + (w - grp * pairs);
    it = P.causal ? (P.n_it - 1 - grp) : grp;
    b = bh / P.H;
    h = bh - b * P.H;
    int row_end = min(P.T, (it + 1) * kBM);  // exclusive
    njt = P.causal ? ((row_end - 1) / kBN + 1) : ((P.T + kBN - 1) / kBN);
}

// The i-th item of round r for this CTA: rounds are dealt in snake order
// (forward, then backward), which pairs heavy with light causal items.
MC_D int item_of_round(int r) {
    const int c = (r & 1) ? (int)(gridDim.x - 1 - blockIdx.x) : (int)blockIdx.x;
    return r * (int)gridDim.x + c;
}

__global__ void __launch_bounds__(kScanThreads, 1) scan_kernel(const __grid_constant__ ScanParams P) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    static_assert(sizeof(ScanSmemTail) <= 1024, "tail");
    ScanSmemTail* tail = reinterpret_cast<ScanSmemTail*>(smem);
    const int nkb = P.nkb_main + P.nkb_rope;
    const int nst = P.stages;
    uint8_t* sQ = smem + 1024;                        // Q buffer qb, block kb: sQ + (qb * nkb + kb) * 16 KB
    uint8_t* sK = sQ + 2 * nkb * kQBlockBytes;
    volatile int* abort_flag = &tail->abort_flag;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < nst; ++s) {
            mbar_init(&tail->kfull[s], 1);
            mbar_init(&tail->kempty[s], 1);
        }
        for (int qb = 0; qb < 2; ++qb) {
            mbar_init(&tail->qfull[qb], 1);
            mbar_init(&tail->qempty[qb], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&tail->tfull[a], 1);
            mbar_init(&tail->tempty[a], 4);
        }
        mbar_init(&tail->drain, 1);
        tail->abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&P.tmQ);
        tma_prefetch_desc(&P.tmK);
        if (P.nkb_rope) tma_prefetch_desc(&P.tmKR);
    }
    if (warp == 1) {
        tmem_alloc(&tail->tmem_base, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = tail->tmem_base;
    pdl_wait();

    if (warp == 0) {
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t issued[kScanMaxStages] = {0, 0, 0, 0, 0, 0};
            uint32_t n = 0;  // items started by this CTA: Q buffer n & 1
            bool ok = true;
            for (int r = 0, i = item_of_round(0); i < P.total_items && ok; i = item_of_round(++r), ++n) {
                int b, h, it, njt;
                decode_item(P, i, b, h, it, njt);
                const int qb = n & 1;
                if (!mbar_wait(&tail->qempty[qb], ((n >> 1) & 1) ^ 1, abort_flag, P.status)) break;
                mbar_arrive_expect_tx(&tail->qfull[qb], nkb * kQBlockBytes);
                for (int kb = 0; kb < nkb; ++kb)
                    tma_load_3d(sQ + (qb * nkb + kb) * kQBlockBytes, &P.tmQ, &tail->qfull[qb],
                                h * P.q_head_stride + kb * kBK, it * kBM, b);
                for (int jt = 0; jt < njt && ok; ++jt) {
                    for (int kb = 0; kb < nkb; ++kb) {
                        if (!mbar_wait(&tail->kempty[stage], phase ^ 1, abort_flag, P.status)) {
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(&tail->kfull[stage], kKStageBytes);
                        if (kb < P.nkb_main)
                            tma_load_3d(sK + stage * kKStageBytes, &P.tmK, &tail->kfull[stage],
                                        h * P.k_head_stride + kb * kBK, jt * kBN, b);
                        else
                            tma_load_3d(sK + stage * kKStageBytes, &P.tmKR, &tail->kfull[stage],
                                        P.kr_col, jt * kBN, b);
                        ++issued[stage];
                        if (++stage == nst) {
                            stage = 0;
                            phase ^= 1;
                        }
                    }
                }
            }
            volatile int never = 0;
            for (int s = 0; s < nst; ++s)
                if (issued[s]) mbar_wait(&tail->kfull[s], (issued[s] - 1) & 1, &never, P.status);
            // Q buffer qb was last filled by item n-1 (qb = (n-1)&1) or n-2
            for (uint32_t j = (n > 2 ? n - 2 : 0); j < n; ++j)
                mbar_wait(&tail->qfull[j & 1], (j >> 1) & 1, &never, P.status);
        }
    } else if (warp == 1) {
        int stage = 0, acc = 0;
        uint32_t phase = 0, aphase = 0;
        uint32_t n = 0;
        bool ok = true;
        const uint32_t idesc = idesc_f16kind(kBM, kBN, 0, 1);  // fp16 Q and K
        for (int r = 0, i = item_of_round(0); i < P.total_items && ok; i = item_of_round(++r), ++n) {
            int b, h, it, njt;
            decode_item(P, i, b, h, it, njt);
            const int qb = n & 1;
            const uint32_t q0 = smem_u32(sQ + qb * nkb * kQBlockBytes);
            if (!mbar_wait(&tail->qfull[qb], (n >> 1) & 1, abort_flag, P.status)) break;
            tc_fence_after();
            for (int jt = 0; jt < njt && ok; ++jt) {
                if (!mbar_wait(&tail->tempty[acc], aphase ^ 1, abort_flag, P.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * kBN);
                for (int kb = 0; kb < nkb; ++kb) {
                    if (!mbar_wait(&tail->kfull[stage], phase, abort_flag, P.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    if (lane == 0) {
                        const uint32_t k0 = smem_u32(sK + stage * kKStageBytes);
                        const uint32_t qa = q0 + kb * kQBlockBytes;
#pragma unroll
                        for (int k = 0; k < kBK / 16; ++k)
                            umma_bf16(d_tmem, sw128_desc(qa + k * 32, 16, 1024),
                                      sw128_desc(k0 + k * 32, 16, 1024), idesc, (kb | k) != 0);
                        umma_commit(&tail->kempty[stage]);
                    }
                    __syncwarp();
                    if (++stage == nst) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
                if (!ok) break;
                if (lane == 0) umma_commit(&tail->tfull[acc]);
                __syncwarp();
                if (++acc == 2) {
                    acc = 0;
                    aphase ^= 1;
                }
            }
            if (!ok) break;
            if (lane == 0) umma_commit(&tail->qempty[qb]);  // Q buffer reusable once these MMAs finish
            __syncwarp();
        }
        if (lane == 0) umma_commit(&tail->drain);
        __syncwarp();
        volatile int never = 0;
        mbar_wait(&tail->drain, 0, &never, P.status);
    } else {
        const int quarter = warp & 3;
        int acc = 0;
        uint32_t aphase = 0;
        bool ok = true;
        for (int r = 0, i = item_of_round(0); i < P.total_items && ok; i = item_of_round(++r)) {
            int b, h, it, njt;
            decode_item(P, i, b, h, it, njt);
            const int row = it * kBM + quarter * 32 + lane;
            const int tile_row0 = it * kBM;
            const bool rows_full = tile_row0 + kBM <= P.T;
            float m0 = -INFINITY, m1 = -INFINITY, m2 = -INFINITY, m3 = -INFINITY;
            for (int jt = 0; jt < njt; ++jt) {
                if (!mbar_wait(&tail->tfull[acc], aphase, abort_flag, P.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const int col_base = jt * kBN;
                const bool full = rows_full && (col_base + kBN <= P.T) &&
                                  (!P.causal || col_base + kBN - 1 <= tile_row0);
                const uint32_t tbase = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * kBN);
#pragma unroll 1
                for (int half = 0; half < 2; ++half) {
                    uint32_t v[128];
                    tmem_ld32(tbase + half * 128, v);
                    tmem_ld32(tbase + half * 128 + 32, v + 32);
                    tmem_ld32(tbase + half * 128 + 64, v + 64);
                    tmem_ld32(tbase + half * 128 + 96, v + 96);
                    tmem_ld_wait();
                    if (full) {
#pragma unroll
                        for (int e = 0; e < 128; e += 8) {
                            m0 = max3_nan(m0, __uint_as_float(v[e]), __uint_as_float(v[e + 1]));
                            m1 = max3_nan(m1, __uint_as_float(v[e + 2]), __uint_as_float(v[e + 3]));
                            m2 = max3_nan(m2, __uint_as_float(v[e + 4]), __uint_as_float(v[e + 5]));
                            m3 = max3_nan(m3, __uint_as_float(v[e + 6]), __uint_as_float(v[e + 7]));
                        }
                    } else {
                        const int c0 = col_base + half * 128;
                        const int lim = P.causal ? min(row + 1, P.T) : P.T;  // valid cols < lim
                        const bool row_ok = row < P.T;
#pragma unroll
                        for (int e = 0; e < 128; e += 2) {
                            float a = (row_ok && c0 + e < lim) ? __uint_as_float(v[e]) : -INFINITY;
                            float c = (row_ok && c0 + e + 1 < lim) ? __uint_as_float(v[e + 1]) : -INFINITY;
                            if (e & 2) m1 = max3_nan(m1, a, c);
                            else m0 = max3_nan(m0, a, c);
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&tail->tempty[acc]);
                if (++acc == 2) {
                    acc = 0;
                    aphase ^= 1;
                }
            }
            if (!ok) break;
            float m = warp_max_nan(max_nan(max_nan(m0, m1), max_nan(m2, m3)));
            if (lane == 0 && m != -INFINITY)  // -inf: every row of this warp is past T
                merge_smax(m, P.sqrt_d, P.s_max, P.s_bh, b, P.H, h, P.status);
        }
    }

    pdl_trigger();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_base, 512);
}

cudaError_t launch_scan(const ScanArgs& a, cudaStream_t stream) {
    ScanParams P;
    memset(&P, 0, sizeof(P));
    const int nkb = a.nkb_main + a.nkb_rope;
    if (nkb < 1 || nkb > kScanQBlocks) return cudaErrorInvalidValue;
    // Q rows hold every head: [B][T][q_ld]; the item's tile is box {64, 128}
    if (!make_tmap_3d(&P.tmQ, a.q, a.q_ld, a.T, a.B, a.q_ld, (uint64_t)a.q_ld * a.T, kBK, kBM, 1))
        return cudaErrorInvalidValue;
    if (!make_tmap_3d(&P.tmK, a.k, a.k_ld, a.T, a.B, a.k_ld, (uint64_t)a.k_ld * a.T, kBK, kBN, 1))
        return cudaErrorInvalidValue;
    if (a.nkb_rope) {
        if (!make_tmap_3d(&P.tmKR, a.kr, a.kr_ld, a.T, a.B, a.kr_ld, (uint64_t)a.kr_ld * a.T, kBK, kBN, 1))
            return cudaErrorInvalidValue;
    } else {
        P.tmKR = P.tmK;
    }
    P.B = a.B;
    P.T = a.T;
    P.H = a.H;
    P.causal = a.causal;
    P.q_head_stride = a.q_head_stride;
    P.k_head_stride = a.k_head_stride;
    P.nkb_main = a.nkb_main;
    P.nkb_rope = a.nkb_rope;
    P.kr_col = a.kr_col;
    P.n_it = (a.T + kBM - 1) / kBM;
    P.total_items = a.B * a.H * P.n_it;
    P.sqrt_d = sqrtf(a.d);
    P.s_max = a.s_max;
    P.s_bh = a.s_bh;
    P.status = device_status_ptr();
    static bool attr_set[64] = {false};
    int dev = current_device();
    if (dev < 0) return cudaErrorInvalidDevice;
    if (dev < 64 && !attr_set[dev]) {
        cudaError_t e = cudaFuncSetAttribute(scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kScanSmem);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    int grid = num_sms();
    if (grid > P.total_items) grid = P.total_items;
    // Launches of at most 16 rounds: one band, so the heavy-first order spans
    // the whole launch and balances the causal tail ([2, 8192, 16 heads]
    // causal: 0.197 ms against 0.208 with one round per band and 0.227 with
    // four).  Longer launches: about one round of items per band, whose K
    // tiles then stay in L2 (K2 MLA layer and long-context scan 2.6-3.4%
    // faster than with two rounds, 3.5-4.6% faster than with sixteen).
    if (P.total_items <= 16 * grid)
        P.band = a.B * a.H;
    else
        P.band = std::max(1, std::min(a.B * a.H, (grid + P.n_it - 1) / P.n_it));
    P.stages = std::min(kScanMaxStages, (kScanRing - 2 * nkb * kQBlockBytes) / kKStageBytes);
    TraceScope ts("scan", stream);
    return launch_pdl(scan_kernel, dim3(grid), dim3(kScanThreads), kScanSmem, stream, P);
}

// ---------------------------------------------------------------------------
// CUDA-core fp32 path for small or unaligned MHA shapes
// ---------------------------------------------------------------------------
template <typename T>
MC_D float load_f(const T* p, size_t i);
template <>
MC_D float load_f<float>(const float* p, size_t i) { return p[i]; }
template <>
MC_D float load_f<__nv_bfloat16>(const __nv_bfloat16* p, size_t i) { return __bfloat162float(p[i]); }

template <typename T>
__global__ void proj_simt_kernel(const T* __restrict__ x, const T* __restrict__ w, float* __restrict__ out,
                                 int rows, int D, int N) {
    pdl_wait();
    size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= (size_t)rows * N) return;
    int r = (int)(idx / N), c = (int)(idx % N);
    float s = 0.f;
    for (int k = 0; k < D; ++k) s = fmaf(load_f(x, (size_t)r * D + k), load_f(w, (size_t)k * N + c), s);
    out[idx] = s;
    pdl_trigger();
}

cudaError_t launch_proj_simt(const void* x, const void* w, mc_dtype dt, float* out, int rows, int D,
                             int N, cudaStream_t stream) {
    size_t n = (size_t)rows * N;
    int threads = 256;
    unsigned blocks = (unsigned)((n + threads - 1) / threads);
    TraceScope ts("proj_simt", stream);
    if (dt == MC_F32)
        return launch_pdl(proj_simt_kernel<float>, dim3(blocks), dim3(threads), 0, stream, (const float*)x,
                          (const float*)w, out, rows, D, N);
    return launch_pdl(proj_simt_kernel<__nv_bfloat16>, dim3(blocks), dim3(threads), 0, stream,
                      (const __nv_bfloat16*)x, (const __nv_bfloat16*)w, out, rows, D, N);
}

// one thread per (b, h, i): max over j of q_i . k_j (fp32), q/k [B*T][H*dh]
__global__ void scan_simt_kernel(const float* __restrict__ q, const float* __restrict__ k, int B, int T,
                                 int H, int dh, int causal, unsigned* __restrict__ keys) {
    pdl_wait();
    size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= (size_t)B * H * T) return;
    int i = (int)(idx % T);
    int bh = (int)(idx / T);
    int h = bh % H, b = bh / H;
    const size_t ld = (size_t)H * dh;
    const float* qi = q + ((size_t)b * T + i) * ld + (size_t)h * dh;
    float m = -INFINITY;
    int jend = causal ? i + 1 : T;
    for (int j = 0; j < jend; ++j) {
        const float* kj = k + ((size_t)b * T + j) * ld + (size_t)h * dh;
        float s = 0.f;
        for (int f = 0; f < dh; ++f) s = fmaf(qi[f], kj[f], s);
        m = max_nan(m, s);
    }
    atomicMax(&keys[b * H + h], float_key(m));
    pdl_trigger();
}

cudaError_t launch_scan_simt(const float* q, const float* k, int B, int T, int H, int dh, int causal,
                             unsigned* keys, cudaStream_t stream) {
    size_t n = (size_t)B * H * T;
    int threads = 128;
    unsigned blocks = (unsigned)((n + threads - 1) / threads);
    TraceScope ts("scan_simt", stream);
    return launch_pdl(scan_simt_kernel, dim3(blocks), dim3(threads), 0, stream, q, k, B, T, H, dh, causal, keys);
}

// ---------------------------------------------------------------------------
// keys -> S_max
// ---------------------------------------------------------------------------
__global__ void finalize_smax_kernel(const unsigned* __restrict__ keys, int B, int H, float sqrt_d,
                                     int accumulate, float* __restrict__ s_max, float* __restrict__ s_bh,
                                     unsigned* status) {
    pdl_wait();
    int h = blockIdx.x * blockDim.x + threadIdx.x;
    if (h >= H) return;
    finalize_head(keys, B, H, h, sqrt_d, accumulate, s_max, s_bh, status);
    pdl_trigger();
}

cudaError_t launch_finalize_smax(const unsigned* keys, int B, int H, float d, int accumulate, float* s_max,
                                 float* s_bh, cudaStream_t stream) {
    int threads = 64;
    int blocks = (H + threads - 1) / threads;
    TraceScope ts("finalize_smax", stream);
    return launch_pdl(finalize_smax_kernel, dim3(blocks), dim3(threads), 0, stream, keys, B, H, sqrtf(d),
                      accumulate, s_max, s_bh, device_status_ptr());
}

// (cos, sin)(t * base^(-2f/64)).  The angle is formed in double in units of
// pi and reduced exactly to [-1, 1] (subtracting an even integer is exact),
// so positions up to the longest sequences keep float accuracy; one float
// sincospi per entry then does the rest.
__global__ void rope_table_kernel(float2* tab, int T, double base) {
    __shared__ double th[32];  // theta_f / pi
    if (threadIdx.x < 32) th[threadIdx.x] = pow(base, -2.0 * (double)threadIdx.x / 64.0) / M_PI;
    __syncthreads();
    pdl_wait();
    int idx = blockIdx.x * blockDim.x + threadIdx.x;
    if (idx < T * 32) {
        int t = idx >> 5, f = idx & 31;
        double x = (double)t * th[f];
        x -= 2.0 * rint(0.5 * x);
        float sn, cs;
        sincospif((float)x, &sn, &cs);
        tab[idx] = make_float2(cs, sn);
    }
    pdl_trigger();
}

cudaError_t launch_rope_table(float2* tab, int T, float base, cudaStream_t stream) {
    int threads = 256;
    int blocks = (T * 32 + threads - 1) / threads;
    TraceScope ts("rope_table", stream);
    return launch_pdl(rope_table_kernel, dim3(blocks), dim3(threads), 0, stream, tab, T, (double)base);
}

}  // namespace mc
