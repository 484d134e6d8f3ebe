// elementwise.cu -- HBM-bound passes of the MuonClip step (sm_103a):
//   * QK-Clip column-block scaling (MHA, MLA, global), one rounding per weight
//   * Muon momentum + bf16 cast of the Newton-Schulz input (transposed for
//     tall matrices) with a deterministic per-tile sum of squares
//   * Frobenius-norm finalisation
//   * the RMS-matched, weight-decayed update W <- W - lr (rms O + wd W)
//   * the self-test of the bounded on-chip waits (one small CTA)
// All loads and stores are 128-bit where the layout allows.
#include "common.cuh"
#include "internal.h"

namespace mc {

// ---------------------------------------------------------------------------
// QK-Clip
// ---------------------------------------------------------------------------

// gamma = min(1, tau / s), 1 when s is not > 0 (the K2 review's gamma
// equation and its reference's where(before > 0, tau / before, 1)).
MC_D float clip_gamma(float s, float tau) {
    if (!(s > 0.0f)) return 1.0f;
    return fminf(1.0f, __fdiv_rn(tau, s));
}

// Product w * f rounded to odd in float (Boldo & Melquiond, "Emulation of
// FMA and correctly rounded sums: proved algorithms using rounding to odd",
// 2008): p = RN(w f), e = w f - p exactly (fma); when e != 0 the result is
// the truncation of w f with its last bit forced to 1.  A later RN to bf16
// (8 < 24 - 1 bits) then equals one rounding of the exact product.
MC_D float mul_round_odd(float w, float f) {
    float p = __fmul_rn(w, f);
    float e = __fmaf_rn(w, f, -p);
    if (e != 0.0f) {
        uint32_t u = __float_as_uint(p);
        if ((e < 0.0f) != (p < 0.0f)) u -= 1u;  // |p| > |w f|: step toward zero
        u |= 1u;
        p = __uint_as_float(u);
    }
    return p;
}

MC_D void scale8_bf16(__nv_bfloat16* p, float f) {
    uint4 u = *reinterpret_cast<const uint4*>(p);
    __nv_bfloat16* h = reinterpret_cast<__nv_bfloat16*>(&u);
#pragma unroll
    for (int i = 0; i < 8; ++i) h[i] = __float2bfloat16_rn(mul_round_odd(__bfloat162float(h[i]), f));
    *reinterpret_cast<uint4*>(p) = u;
}
MC_D void scale8_f32(float* p, float f) {
    float4 a = *reinterpret_cast<const float4*>(p);
    float4 b = *reinterpret_cast<const float4*>(p + 4);
    a.x = __fmul_rn(a.x, f); a.y = __fmul_rn(a.y, f); a.z = __fmul_rn(a.z, f); a.w = __fmul_rn(a.w, f);
    b.x = __fmul_rn(b.x, f); b.y = __fmul_rn(b.y, f); b.z = __fmul_rn(b.z, f); b.w = __fmul_rn(b.w, f);
    *reinterpret_cast<float4*>(p) = a;
    *reinterpret_cast<float4*>(p + 4) = b;
}

// grid (H, nseg, chunks): block (h, s) scales head h's columns of segment s
__global__ void clip_kernel(const ClipArgs a) {
    pdl_wait();
    const int h = blockIdx.x;
    const ClipSeg& sg = a.seg[blockIdx.y];
    const float g = clip_gamma(a.s_max[h], a.tau);
    if (a.gamma_out && blockIdx.y == 0 && blockIdx.z == 0 && threadIdx.x == 0) a.gamma_out[h] = g;
    if (g == 1.0f) return;  // unclipped head: never written
    const float f = sg.use_gamma ? g : __fsqrt_rn(g);
    const long long col = (long long)sg.col0 + (long long)h * sg.head_stride;
    const bool vec = ((sg.ld | col | sg.width) & 7) == 0 && (reinterpret_cast<uintptr_t>(sg.w) & 15) == 0;
    if (vec) {
        const int per_row = sg.width >> 3;
        const long long n = (long long)sg.rows * per_row;
        for (long long i = (long long)blockIdx.z * blockDim.x + threadIdx.x; i < n;
             i += (long long)gridDim.z * blockDim.x) {
            long long r = i / per_row;
            int v = (int)(i - r * per_row);
            long long off = r * sg.ld + col + 8 * v;
            if (a.bf16) scale8_bf16(reinterpret_cast<__nv_bfloat16*>(sg.w) + off, f);
            else scale8_f32(reinterpret_cast<float*>(sg.w) + off, f);
        }
        pdl_trigger();
    } else {
        const long long n = (long long)sg.rows * sg.width;
        for (long long i = (long long)blockIdx.z * blockDim.x + threadIdx.x; i < n;
             i += (long long)gridDim.z * blockDim.x) {
            long long r = i / sg.width;
            long long off = r * sg.ld + col + (i - r * sg.width);
            if (a.bf16) {
                __nv_bfloat16* p = reinterpret_cast<__nv_bfloat16*>(sg.w) + off;
                *p = __float2bfloat16_rn(mul_round_odd(__bfloat162float(*p), f));
            } else {
                float* p = reinterpret_cast<float*>(sg.w) + off;
                *p = __fmul_rn(*p, f);
            }
        }
        pdl_trigger();
    }
}

cudaError_t launch_clip(const ClipArgs& a, cudaStream_t stream) {
    if (a.H <= 0 || a.nseg <= 0) return cudaSuccess;
    long long max_elems = 0;
    for (int s = 0; s < a.nseg; ++s) {
        long long e = (long long)a.seg[s].rows * a.seg[s].width;
        if (e > max_elems) max_elems = e;
    }
    int threads = 256;
    long long chunks = (max_elems / 8 + threads - 1) / threads;
    if (chunks < 1) chunks = 1;
    if (chunks > 64) chunks = 64;
    dim3 grid(a.H, a.nseg, (unsigned)chunks);
    TraceScope ts("clip", stream);
    return launch_pdl(clip_kernel, grid, dim3(threads), 0, stream, a);
}

// Global clip: gamma from max_h s_max[h] (NaN propagates), then every
// element of wq x gamma^alpha and of wk x gamma^(1-alpha).
__global__ void clip_global_kernel(void* wq, void* wk, int bf16, long long n, const float* s_max, int H,
                                   float tau, float alpha, float* gamma_out) {
    pdl_wait();
    float s = s_max[0];
    for (int h = 1; h < H; ++h) s = max_nan(s, s_max[h]);
    const float g = clip_gamma(s, tau);
    if (gamma_out && blockIdx.x == 0 && threadIdx.x == 0) *gamma_out = g;
    if (g == 1.0f) return;
    const float fq = (float)pow((double)g, (double)alpha);
    const float fk = (float)pow((double)g, 1.0 - (double)alpha);
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (long long)gridDim.x * blockDim.x) {
        if (bf16) {
            __nv_bfloat16* q = reinterpret_cast<__nv_bfloat16*>(wq) + i;
            __nv_bfloat16* k = reinterpret_cast<__nv_bfloat16*>(wk) + i;
            *q = __float2bfloat16_rn(mul_round_odd(__bfloat162float(*q), fq));
            *k = __float2bfloat16_rn(mul_round_odd(__bfloat162float(*k), fk));
        } else {
            float* q = reinterpret_cast<float*>(wq) + i;
            float* k = reinterpret_cast<float*>(wk) + i;
            *q = __fmul_rn(*q, fq);
            *k = __fmul_rn(*k, fk);
        }
    }
    pdl_trigger();
}

cudaError_t launch_clip_global(void* wq, void* wk, int bf16, long long n, const float* s_max, int H, float tau,
                               float alpha, float* gamma_out, cudaStream_t stream) {
    int threads = 256;
    long long blocks = (n + threads - 1) / threads;
    if (blocks > 4096) blocks = 4096;
    if (blocks < 1) blocks = 1;
    TraceScope ts("clip_global", stream);
    return launch_pdl(clip_global_kernel, dim3((unsigned)blocks), dim3(threads), 0, stream, wq, wk, bf16, n,
                      s_max, H, tau, alpha, gamma_out);
}

// ---------------------------------------------------------------------------
// bf16 -> fp16 (weights feeding an fp16 contraction)
// ---------------------------------------------------------------------------
__global__ void bf16_to_f16_kernel(const __nv_bfloat16* __restrict__ src, __half* __restrict__ dst, long long n) {
    pdl_wait();
    const long long nv = n / 8;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < nv; i += (long long)gridDim.x * blockDim.x) {
        uint4 u = reinterpret_cast<const uint4*>(src)[i];
        const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&u);
        uint4 o;
        __half2* h = reinterpret_cast<__half2*>(&o);
#pragma unroll
        for (int k = 0; k < 4; ++k) h[k] = __float22half2_rn(__bfloat1622float2(b[k]));
        reinterpret_cast<uint4*>(dst)[i] = o;
    }
    for (long long i = nv * 8 + (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (long long)gridDim.x * blockDim.x)
        dst[i] = __float2half_rn(__bfloat162float(src[i]));
    pdl_trigger();
}

cudaError_t launch_bf16_to_f16(const void* src, void* dst, long long n, cudaStream_t stream) {
    if (n <= 0) return cudaSuccess;
    int threads = 256;
    long long blocks = (n / 8 + threads - 1) / threads;
    if (blocks < 1) blocks = 1;
    if (blocks > (long long)num_sms() * 8) blocks = (long long)num_sms() * 8;
    TraceScope ts("to_f16", stream);
    return launch_pdl(bf16_to_f16_kernel, dim3((unsigned)blocks), dim3(threads), 0, stream,
                      (const __nv_bfloat16*)src, (__half*)dst, n);
}

// ---------------------------------------------------------------------------
// Muon passes over 64 x 64 tiles of X (the Newton-Schulz orientation)
// ---------------------------------------------------------------------------

// W <- W - lr (rms O + wd W) ("Notes on Moonlight", "Scaling up Muon"),
// every product and sum rounded once in the order written.  The tiled pass
// and the flat pass over a ZeRO-1 shard share it, so a sharded update
// matches the whole-matrix one bit for bit.
MC_D float muon_update_elem(float w, float o, float lr, float rms, float wd) {
    return __fsub_rn(w, __fmul_rn(lr, __fadd_rn(__fmul_rn(rms, o), __fmul_rn(wd, w))));
}

constexpr int kTile = 64;
constexpr int kMatThreads = 256;

MC_D void find_mat(const MatBatch& B, int t, int& di) {
    di = 0;
    while (di + 1 < B.count && t >= B.d[di + 1].tile_begin) ++di;
}

// The CTA's sum of the threads' partial sums of squares, in fp64 and in a
// fixed order (lanes by butterfly, then warps in turn), stored at *out.
MC_D void block_sumsq(float ss, double* red, double* out) {
    const int tid = threadIdx.x;
    double s = (double)ss;
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, o);
    if ((tid & 31) == 0) red[tid >> 5] = s;
    __syncthreads();
    if (tid == 0) {
        double tot = 0.0;
        for (int w = 0; w < kMatThreads / 32; ++w) tot += red[w];
        *out = tot;
    }
    __syncthreads();
}

// Source element (r, c) of the [rows][cols] matrix <-> X element (i, j):
// X = S^T when tr, else X = S.
__global__ void __launch_bounds__(kMatThreads) mat_pass_kernel(const __grid_constant__ MatBatch B) {
    __shared__ float U[kTile][kTile + 1];
    __shared__ double red[kMatThreads / 32];
    const int tid = threadIdx.x;
    pdl_wait();
    if (B.info && B.mode <= 1 && blockIdx.x == 0 && tid < B.count) {
        const MatDesc& d = B.d[tid];
        MatInfo mi;
        mi.partial = d.partial;
        mi.nparts = (d.m_pad / kTile) * (d.n_pad / kTile);
        mi.pad_ = 0;
        B.info[B.info_base + tid] = mi;
    }
    for (int t = blockIdx.x; t < B.total_tiles; t += gridDim.x) {
        int di;
        find_mat(B, t, di);
        const MatDesc& d = B.d[di];
        const int local = t - d.tile_begin;
        const int ti = local / d.tiles_x, tj = local - ti * d.tiles_x;
        const int i0 = ti * kTile, j0 = tj * kTile;  // X tile origin
        // the matching source tile: rows [sr0, sr0+64), cols [sc0, sc0+64)
        const int sr0 = d.tr ? j0 : i0, sc0 = d.tr ? i0 : j0;
        const int m = d.tr ? d.cols : d.rows, n = d.tr ? d.rows : d.cols;
        const bool any = i0 < m && j0 < n;

        // flat matrices: X has the source's own layout (no transpose, no
        // padding), so chunk `local` is 4096 consecutive elements of both and
        // each warp streams whole 512-byte runs; the chunks take the places of
        // the tiles (one sum of squares each)
        const size_t fbase = (size_t)local * (kTile * kTile) + tid * 4;

        if (B.mode <= 1 && d.flat) {
            float ss = 0.f;
#pragma unroll 1
            for (int p = 0; p < 4; ++p) {
                const size_t off = fbase + (size_t)p * (kMatThreads * 4);
                float4 u = *reinterpret_cast<const float4*>(d.m + off);
                if (B.mode == 0) {
                    const float4 gv = *reinterpret_cast<const float4*>(d.g + off);
                    float4 mv;
                    mv.x = __fmaf_rn(B.mu, u.x, gv.x);
                    mv.y = __fmaf_rn(B.mu, u.y, gv.y);
                    mv.z = __fmaf_rn(B.mu, u.z, gv.z);
                    mv.w = __fmaf_rn(B.mu, u.w, gv.w);
                    *reinterpret_cast<float4*>(d.m + off) = mv;
                    u = B.nesterov ? make_float4(__fmaf_rn(B.mu, mv.x, gv.x), __fmaf_rn(B.mu, mv.y, gv.y),
                                                 __fmaf_rn(B.mu, mv.z, gv.z), __fmaf_rn(B.mu, mv.w, gv.w))
                                   : mv;
                }
                ss += u.x * u.x + u.y * u.y + u.z * u.z + u.w * u.w;
                __nv_bfloat162 h0 = __floats2bfloat162_rn(u.x, u.y);
                __nv_bfloat162 h1 = __floats2bfloat162_rn(u.z, u.w);
                uint2 pk;
                pk.x = *reinterpret_cast<uint32_t*>(&h0);
                pk.y = *reinterpret_cast<uint32_t*>(&h1);
                *reinterpret_cast<uint2*>(d.x + off) = pk;
            }
            block_sumsq(ss, red, d.partial + local);
        } else if (d.flat) {
            const float osc = d.oscale ? *d.oscale : 1.0f;
#pragma unroll 1
            for (int p = 0; p < 4; ++p) {
                const size_t off = fbase + (size_t)p * (kMatThreads * 4);
                uint2 pk = *reinterpret_cast<const uint2*>(d.x + off);
                float2 a, b;
                if (B.x_f16) {
                    a = __half22float2(*reinterpret_cast<__half2*>(&pk.x));
                    b = __half22float2(*reinterpret_cast<__half2*>(&pk.y));
                } else {
                    a = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&pk.x));
                    b = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&pk.y));
                }
                const float o0 = osc * a.x, o1 = osc * a.y, o2 = osc * b.x, o3 = osc * b.y;
                if (B.mode == 2) {
                    float4 w = *reinterpret_cast<const float4*>(d.w + off);
                    w.x = muon_update_elem(w.x, o0, B.lr, d.rms, B.wd);
                    w.y = muon_update_elem(w.y, o1, B.lr, d.rms, B.wd);
                    w.z = muon_update_elem(w.z, o2, B.lr, d.rms, B.wd);
                    w.w = muon_update_elem(w.w, o3, B.lr, d.rms, B.wd);
                    *reinterpret_cast<float4*>(d.w + off) = w;
                } else {
                    *reinterpret_cast<float4*>(d.w + off) = make_float4(o0, o1, o2, o3);
                }
            }
        } else if (B.mode <= 1) {
            // ---- momentum (+ Nesterov) and cast: source -> U -> X ----
            float ss = 0.f;
            if (any) {
#pragma unroll
                for (int p = 0; p < 4; ++p) {
                    const int lr = p * 16 + (tid >> 4), lc = (tid & 15) * 4;
                    const int r = sr0 + lr, c = sc0 + lc;
                    float4 u = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (r < d.rows && c < d.cols && !d.vec) {
                        // any width: element by element, zero past the last column
                        float uu[4];
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            uu[k] = 0.f;
                            if (c + k < d.cols) {
                                const size_t off = (size_t)r * d.cols + c + k;
                                float mv = d.m[off];
                                if (B.mode == 0) {
                                    const float gv = d.g[off];
                                    mv = __fmaf_rn(B.mu, mv, gv);
                                    d.m[off] = mv;
                                    uu[k] = B.nesterov ? __fmaf_rn(B.mu, mv, gv) : mv;
                                } else {
                                    uu[k] = mv;
                                }
                            }
                        }
                        u = make_float4(uu[0], uu[1], uu[2], uu[3]);
                    } else if (r < d.rows && c < d.cols) {
                        const size_t off = (size_t)r * d.cols + c;
                        float4 mv = *reinterpret_cast<const float4*>(d.m + off);
                        if (B.mode == 0) {
                            float4 gv = *reinterpret_cast<const float4*>(d.g + off);
                            mv.x = __fmaf_rn(B.mu, mv.x, gv.x);
                            mv.y = __fmaf_rn(B.mu, mv.y, gv.y);
                            mv.z = __fmaf_rn(B.mu, mv.z, gv.z);
                            mv.w = __fmaf_rn(B.mu, mv.w, gv.w);
                            *reinterpret_cast<float4*>(d.m + off) = mv;
                            if (B.nesterov) {
                                u = make_float4(__fmaf_rn(B.mu, mv.x, gv.x), __fmaf_rn(B.mu, mv.y, gv.y),
                                                __fmaf_rn(B.mu, mv.z, gv.z), __fmaf_rn(B.mu, mv.w, gv.w));
                            } else {
                                u = mv;
                            }
                        } else {
                            u = mv;
                        }
                    }
                    ss += u.x * u.x + u.y * u.y + u.z * u.z + u.w * u.w;
                    U[lr][lc] = u.x;
                    U[lr][lc + 1] = u.y;
                    U[lr][lc + 2] = u.z;
                    U[lr][lc + 3] = u.w;
                }
            }
            __syncthreads();
            // write X rows i0.., 4 consecutive j per thread (zeros in padding)
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                const int li = p * 16 + (tid >> 4), lj = (tid & 15) * 4;
                float v[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) v[k] = any ? (d.tr ? U[lj + k][li] : U[li][lj + k]) : 0.f;
                __nv_bfloat162 h0 = __floats2bfloat162_rn(v[0], v[1]);
                __nv_bfloat162 h1 = __floats2bfloat162_rn(v[2], v[3]);
                uint2 pk;
                pk.x = *reinterpret_cast<uint32_t*>(&h0);
                pk.y = *reinterpret_cast<uint32_t*>(&h1);
                *reinterpret_cast<uint2*>(d.x + (size_t)(i0 + li) * d.n_pad + j0 + lj) = pk;
            }
            block_sumsq(ss, red, d.partial + local);  // deterministic tile sum of squares
        } else {
            // ---- X -> U -> update W (mode 2) or write O (mode 3) ----
            if (!any) continue;
            const float osc = d.oscale ? *d.oscale : 1.0f;
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                const int li = p * 16 + (tid >> 4), lj = (tid & 15) * 4;
                uint2 pk = *reinterpret_cast<const uint2*>(d.x + (size_t)(i0 + li) * d.n_pad + j0 + lj);
                float2 a, b;
                if (B.x_f16) {
                    a = __half22float2(*reinterpret_cast<__half2*>(&pk.x));
                    b = __half22float2(*reinterpret_cast<__half2*>(&pk.y));
                } else {
                    a = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&pk.x));
                    b = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&pk.y));
                }
                U[li][lj] = a.x;
                U[li][lj + 1] = a.y;
                U[li][lj + 2] = b.x;
                U[li][lj + 3] = b.y;
            }
            __syncthreads();
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                const int lr = p * 16 + (tid >> 4), lc = (tid & 15) * 4;
                const int r = sr0 + lr, c = sc0 + lc;
                if (r < d.rows && c < d.cols) {
                    float o[4];
#pragma unroll
                    for (int k = 0; k < 4; ++k) o[k] = osc * (d.tr ? U[lc + k][lr] : U[lr][lc + k]);
                    const size_t off = (size_t)r * d.cols + c;
                    if (!d.vec) {
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            if (c + k >= d.cols) break;
                            if (B.mode == 2) {
                                d.w[off + k] = muon_update_elem(d.w[off + k], o[k], B.lr, d.rms, B.wd);
                            } else {
                                d.w[off + k] = o[k];
                            }
                        }
                    } else if (B.mode == 2) {
                        float4 w = *reinterpret_cast<const float4*>(d.w + off);
                        w.x = muon_update_elem(w.x, o[0], B.lr, d.rms, B.wd);
                        w.y = muon_update_elem(w.y, o[1], B.lr, d.rms, B.wd);
                        w.z = muon_update_elem(w.z, o[2], B.lr, d.rms, B.wd);
                        w.w = muon_update_elem(w.w, o[3], B.lr, d.rms, B.wd);
                        *reinterpret_cast<float4*>(d.w + off) = w;
                    } else {
                        *reinterpret_cast<float4*>(d.w + off) = make_float4(o[0], o[1], o[2], o[3]);
                    }
                }
            }
            __syncthreads();
        }
    }
    pdl_trigger();
}

cudaError_t launch_mat_pass(const MatBatch& b, cudaStream_t stream) {
    if (b.total_tiles <= 0) return cudaSuccess;
    int grid = num_sms() * 8;
    if (grid > b.total_tiles) grid = b.total_tiles;
    static const char* names[4] = {"muon_momentum", "ns_cast", "muon_update", "ns_out"};
    TraceScope ts(names[b.mode & 3], stream);
    return launch_pdl(mat_pass_kernel, dim3(grid), dim3(kMatThreads), 0, stream, b);
}

// ---------------------------------------------------------------------------
// Flat passes over one ZeRO-1 shard of a matrix ("Notes on Moonlight",
// "Distributed Muon": the optimizer state is partitioned across the
// data-parallel ranks; momentum and the update are elementwise, so each rank
// applies them to its own block).  Same arithmetic as the tiled passes:
//   momentum  M <- mu M + s G   (s scales a summed gradient to the mean),
//             U = M, or the Nesterov input s G + mu M when requested;
//   update    W <- W - lr (rms O + wd W).
// ---------------------------------------------------------------------------
__global__ void momentum_flat_kernel(float* __restrict__ m, const float* __restrict__ g, float* __restrict__ u,
                                     long long n, float mu, float gs, int nesterov, int vec) {
    pdl_wait();
    const long long stride = (long long)gridDim.x * blockDim.x;
    const long long t0 = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    const long long nv = vec ? n / 4 : 0;
    for (long long i = t0; i < nv; i += stride) {
        float4 mv = reinterpret_cast<const float4*>(m)[i];
        float4 gv = reinterpret_cast<const float4*>(g)[i];
        gv.x = __fmul_rn(gv.x, gs); gv.y = __fmul_rn(gv.y, gs);
        gv.z = __fmul_rn(gv.z, gs); gv.w = __fmul_rn(gv.w, gs);
        mv.x = __fmaf_rn(mu, mv.x, gv.x); mv.y = __fmaf_rn(mu, mv.y, gv.y);
        mv.z = __fmaf_rn(mu, mv.z, gv.z); mv.w = __fmaf_rn(mu, mv.w, gv.w);
        reinterpret_cast<float4*>(m)[i] = mv;
        if (u) {
            float4 uv = mv;
            if (nesterov)
                uv = make_float4(__fmaf_rn(mu, mv.x, gv.x), __fmaf_rn(mu, mv.y, gv.y), __fmaf_rn(mu, mv.z, gv.z),
                                 __fmaf_rn(mu, mv.w, gv.w));
            reinterpret_cast<float4*>(u)[i] = uv;
        }
    }
    for (long long i = nv * 4 + t0; i < n; i += stride) {
        const float gv = __fmul_rn(g[i], gs);
        const float mv = __fmaf_rn(mu, m[i], gv);
        m[i] = mv;
        if (u) u[i] = nesterov ? __fmaf_rn(mu, mv, gv) : mv;
    }
    pdl_trigger();
}

__global__ void update_flat_kernel(float* __restrict__ w, const float* __restrict__ o, long long n, float lr,
                                   float rms, float wd, int vec) {
    pdl_wait();
    const long long stride = (long long)gridDim.x * blockDim.x;
    const long long t0 = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    const long long nv = vec ? n / 4 : 0;
    for (long long i = t0; i < nv; i += stride) {
        float4 wv = reinterpret_cast<const float4*>(w)[i];
        const float4 ov = reinterpret_cast<const float4*>(o)[i];
        wv.x = muon_update_elem(wv.x, ov.x, lr, rms, wd);
        wv.y = muon_update_elem(wv.y, ov.y, lr, rms, wd);
        wv.z = muon_update_elem(wv.z, ov.z, lr, rms, wd);
        wv.w = muon_update_elem(wv.w, ov.w, lr, rms, wd);
        reinterpret_cast<float4*>(w)[i] = wv;
    }
    for (long long i = nv * 4 + t0; i < n; i += stride) w[i] = muon_update_elem(w[i], o[i], lr, rms, wd);
    pdl_trigger();
}

static unsigned flat_blocks(long long n) {
    long long b = (n / 4 + 255) / 256;
    if (b < 1) b = 1;
    if (b > (long long)num_sms() * 8) b = (long long)num_sms() * 8;
    return (unsigned)b;
}

cudaError_t launch_momentum_flat(float* m, const float* g, float* u, long long n, float mu, float gs,
                                 int nesterov, cudaStream_t stream) {
    if (n <= 0) return cudaSuccess;
    const int vec = ((reinterpret_cast<uintptr_t>(m) | reinterpret_cast<uintptr_t>(g) |
                      (u ? reinterpret_cast<uintptr_t>(u) : 0)) & 15) == 0;
    TraceScope ts("muon_momentum_shard", stream);
    return launch_pdl(momentum_flat_kernel, dim3(flat_blocks(n)), dim3(256), 0, stream, m, g, u, n, mu, gs,
                      nesterov, vec);
}

cudaError_t launch_update_flat(float* w, const float* o, long long n, float lr, float rms, float wd,
                               cudaStream_t stream) {
    if (n <= 0) return cudaSuccess;
    const int vec = ((reinterpret_cast<uintptr_t>(w) | reinterpret_cast<uintptr_t>(o)) & 15) == 0;
    TraceScope ts("muon_update_shard", stream);
    return launch_pdl(update_flat_kernel, dim3(flat_blocks(n)), dim3(256), 0, stream, w, o, n, lr, rms, wd, vec);
}

// ---------------------------------------------------------------------------
// Order-preserving int32 keys of fp32 S_max values, so the per-head maximum
// over data-parallel ranks is one all-reduce(MAX) of integers: a < b implies
// key(a) < key(b), -0 sits just below +0, and every NaN maps to the largest
// key, so a NaN max logit on any rank reaches every rank (a float max
// reduction may drop it).  Decoding inverts the map (NaNs come back as one
// quiet NaN).
// ---------------------------------------------------------------------------
MC_D int smax_key(float f) {
    if (f != f) return 0x7FFFFFFF;
    const int b = __float_as_int(f);
    return b >= 0 ? b : (b ^ 0x7FFFFFFF);
}
MC_D float smax_unkey(int k) { return __int_as_float(k >= 0 ? k : (k ^ 0x7FFFFFFF)); }

__global__ void smax_keys_kernel(const float* s, int* keys, const int* kin, float* sout, int n) {
    pdl_wait();
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
        if (s) keys[i] = smax_key(s[i]);
        else sout[i] = smax_unkey(kin[i]);
    }
    pdl_trigger();
}

cudaError_t launch_smax_keys(const float* s, int* keys, const int* kin, float* sout, int n, cudaStream_t stream) {
    if (n <= 0) return cudaSuccess;
    const int blocks = (n + 255) / 256 < 64 ? (n + 255) / 256 : 64;
    TraceScope ts("smax_keys", stream);
    return launch_pdl(smax_keys_kernel, dim3(blocks), dim3(256), 0, stream, s, keys, kin, sout, n);
}

// s = 1 / (||U||_F + eps) from the tile partials, summed in a fixed order
__global__ void norm_finalize_kernel(const __grid_constant__ NormArgs a) {
    pdl_wait();
    const int z = blockIdx.x;
    if (z >= a.count) return;
    __shared__ double red[256];
    double s = 0.0;
    for (int i = threadIdx.x; i < a.nparts[z]; i += blockDim.x) s += a.partial[z][i];
    red[threadIdx.x] = s;
    __syncthreads();
    for (int w = blockDim.x / 2; w > 0; w >>= 1) {
        if (threadIdx.x < w) red[threadIdx.x] += red[threadIdx.x + w];
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        double den = sqrt(red[0]) + (double)a.eps;
        a.s[z] = (float)(1.0 / den);
        a.s2[z] = (float)(1.0 / (den * den));
    }
    pdl_trigger();
}

cudaError_t launch_norm_finalize(const NormArgs& a, cudaStream_t stream) {
    if (a.count <= 0) return cudaSuccess;
    TraceScope ts("norm_finalize", stream);
    return launch_pdl(norm_finalize_kernel, dim3(a.count), dim3(256), 0, stream, a);
}

// ---------------------------------------------------------------------------
// Self-test of the bounded on-chip waits: both warps of one CTA wait on
// mbarriers that nothing arrives on, through the same wait as every kernel
// of the library.  Warp 0 gives up after limit_ns (setting MC_DEV_TIMEOUT and
// the CTA's abort flag); warp 1, with the library's normal limit, must then
// leave through the abort flag.  out[w] = warp w's wait in ns, out[2 + w] = 1
// if its barrier completed (it cannot).  Every path ends: no hang, no fault.
// ---------------------------------------------------------------------------
__global__ void wait_selftest_kernel(uint64_t limit_ns, long long* out, unsigned* status) {
    __shared__ __align__(8) uint64_t bar[2];
    __shared__ int abort_flag;
    pdl_wait();
    if (threadIdx.x == 0) {
        mbar_init(&bar[0], 1);
        mbar_init(&bar[1], 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5;
    const uint64_t t0 = globaltimer_ns();
    const bool done = mbar_wait(&bar[warp], 0, &abort_flag, status, warp == 0 ? limit_ns : kWaitLimitNs);
    const uint64_t t1 = globaltimer_ns();
    if ((threadIdx.x & 31) == 0) {
        out[warp] = (long long)(t1 - t0);
        out[2 + warp] = done ? 1 : 0;
    }
    pdl_trigger();
}

cudaError_t launch_wait_selftest(uint64_t limit_ns, long long* out, cudaStream_t stream) {
    TraceScope ts("selftest_wait", stream);
    return launch_pdl(wait_selftest_kernel, dim3(1), dim3(64), 0, stream, limit_ns, out, device_status_ptr());
}

}  // namespace mc
