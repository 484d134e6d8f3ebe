// gemm.cu -- persistent, warp-specialised tcgen05 GEMM for sm_103a.
//
// Persistent CTAs (or CTA pairs) walk a static round-robin list of output
// tiles drawn from up to four problems per phase (projections of one layer,
// or one Newton-Schulz phase over every matrix of a batch).
//   warps 0, 6  TMA producers: warp 0 loads the A half of every stage, warp
//               6 the B half (bf16 or fp16, 128-byte swizzle, K = 128 per
//               stage in two 64-wide chunks) into a 3-stage ring
//   warp 1      TMEM owner and MMA issuer: 8 x tcgen05.mma (K = 16) per
//               stage, one commit per stage, into one of two fp32 TMEM
//               accumulators
//   warps 2..5  epilogue: tcgen05.ld -> scale / aux / RoPE -> bf16, fp16
//               or f32 global stores (mirrored for symmetric outputs)
// The double-buffered accumulator lets the epilogue of tile t overlap the
// MMAs of tile t+1.  Every wait is bounded (see mbar_wait).
#include "common.cuh"
#include "internal.h"

namespace mc {

// A stage: K = KS in chunks of kBK (one 128-byte swizzle row each).
// Single CTAs (N = 128) take KS = 128, eight MMAs per commit: a commit and
// the producer's wait on it cost about as much as four N = 128 MMAs, so four
// MMAs per commit ran at half the tensor rate at N = 128 (measured).
constexpr int kAChunkBytes = kBM * kBK * 2;            // 16 KB
// warp 0 and warp 6: TMA producers (the A and the B half of every stage:
// one thread issues TMA loads at about half the rate two threads in
// different warps reach); warp 1: MMA issuer; warps 2..5: epilogue
constexpr int kGemmThreads = 224;
// epilogue staging: each epilogue warp stages a 32 x 64 chunk of 16-bit
// values in rows of 72 elements (144 B: 16-byte accesses are bank-conflict
// free) so that every global load/store of the epilogue is a coalesced
// 16-byte access by 8 lanes per 128-byte row segment
constexpr int kStageLd = 72;
// 5 KB per warp (1 KB aligned): also holds a dense 32 x 64 box in the 128-byte
// swizzled layout of the TMA tensor store
constexpr int kEpiWarpBytes = 5120;
static_assert(kEpiWarpBytes >= 32 * kStageLd * 2 && kEpiWarpBytes % 1024 == 0, "staging buffer");

// Offset (16-bit elements) of 16-byte segment v of row r in a warp's staging
// buffer: rows of kStageLd elements (padded: conflict-free), or swizzled
// 128-byte rows (segment v stored at v ^ (r mod 8): conflict-free and the
// layout a SWIZZLE_128B tensor map reads).
MC_D int stage_off(bool swz, int r, int v) { return swz ? r * 64 + ((v ^ (r & 7)) << 3) : r * kStageLd + (v << 3); }
// Tile / pipeline shapes (see the launchers at the end): CTA pairs on
// 256 x 256 tiles, each SM holding 128 rows of A and 128 of B per 64 KB
// stage; single CTAs on 128 x 128 tiles for small Newton-Schulz batches.
// Shared-memory copies of the current and the next phase's problems: the
// roles read the problem fields from here instead of the (large, dynamically
// indexed) kernel parameters, whose constant-cache misses would otherwise sit
// on every phase's critical path.  TMA still reads the tensor maps from the
// parameters.
constexpr int kTailBytes = 384;
constexpr int kProbStageBytes = 2 * kPhaseProbs * (int)sizeof(GemmProblem);
template <int BN, int STAGES, bool PAIR, int KS>
struct TileCfg {
    static constexpr int kKChunks = KS / kBK;
    static constexpr int kAStageBytes = kAChunkBytes * kKChunks;
    // a pair computes a 256 x BN tile: each CTA holds 128 rows of A and BN / 2
    // rows (K-major) or columns (MN-major) of B; the MMA reads both halves
    static constexpr int kTileM = PAIR ? 2 * kBM : kBM;
    static constexpr int kBRows = PAIR ? BN / 2 : BN;
    // K-major B: kKChunks chunks of kBRows rows x 128 bytes; MN-major B:
    // kBRows / 64 column chunks of KS rows x 128 bytes
    static constexpr int kBChunkK = kBRows * kBK * 2;
    static constexpr int kBChunkMN = KS * 128;
    static constexpr int kBStage = kBRows * KS * 2;
    static constexpr int kSmem = STAGES * (kAStageBytes + kBStage) + 4 * kEpiWarpBytes + 1024 + kTailBytes +
                                 64 + kProbStageBytes;
    static constexpr uint32_t kTmemCols = 2 * BN;  // two accumulators
};
template <int STAGES>
struct GemmSmemTail {
    uint64_t full[STAGES];
    uint64_t empty[STAGES];
    uint64_t tfull[2];
    uint64_t tempty[2];
    uint64_t drain;
    uint64_t pairbar[2];  // the epilogue's two pairs of warps (rows 0-63 and 64-127 of a CTA's tile)
    uint32_t tmem_base;
    int abort_flag;
};

// Tile t of a phase -> (problem index within the phase, batch, row block,
// column block); sp holds the phase's np problems.
template <int BN, int TM>
MC_D void decode_tile(const GemmProblem* sp, int np, int t, int& pi, int& z, int& tm, int& tn) {
    if (sp[0].a_shared) {
        // row block tm, then the column tiles of every problem in turn
        const int tn_total = sp[np - 1].tn_off + sp[np - 1].tiles_n;
        tm = t / tn_total;
        const int c = t - tm * tn_total;
        pi = 0;
        while (pi + 1 < np && c >= sp[pi + 1].tn_off) ++pi;
        tn = c - sp[pi].tn_off;
        z = 0;
        return;
    }
    pi = 0;
    while (pi + 1 < np && t >= sp[pi + 1].tile_begin) ++pi;
    const GemmProblem& q = sp[pi];
    int local = t - q.tile_begin;
    z = local / q.tiles_per_batch;
    int r = local - z * q.tiles_per_batch;
    if (!q.sym) {
        tm = r / q.tiles_n;
        tn = r - tm * q.tiles_n;
    } else {
        // row block tm holds the tiles tn >= TM tm / BN (those touching c >= r)
        tm = 0;
        while (true) {
            const int first = (TM * tm) / BN;
            int cnt = q.tiles_n - first;
            if (r < cnt) {
                tn = first + r;
                break;
            }
            r -= cnt;
            ++tm;
        }
    }
}

// Copy phase ph's problems from the kernel parameters into shared memory
// (16-byte pieces spread over threads tid0.. of the CTA).
template <int MAXP>
MC_D void stage_phase(const GemmParamsT<MAXP>& P, int ph, GemmProblem* dst, int tid, int nthr) {
    const int pb = P.phase_prob[ph], pe = P.phase_prob[ph + 1];
    const uint4* src = reinterpret_cast<const uint4*>(&P.p[pb]);
    uint4* d = reinterpret_cast<uint4*>(dst);
    const int n = (pe - pb) * (int)(sizeof(GemmProblem) / 16);
    for (int i = tid; i < n; i += nthr) d[i] = src[i];
}

// Grid-wide barrier between phases of a multi-phase (cooperative) launch:
// every CTA's phase stores are released (gpu scope, and to the async proxy
// that the next phase's TMA loads use) before any CTA proceeds.  Bounded.
template <int MAXP>
MC_D void grid_sync(const GemmParamsT<MAXP>& P, int seq, volatile int* abort_flag, int next_ph,
                    GemmProblem* next_dst) {
    tc_fence_before();
    __syncthreads();
    // the other threads stage the next phase's problems while thread 0 waits
    if (next_ph >= 0 && threadIdx.x >= 32) stage_phase(P, next_ph, next_dst, threadIdx.x - 32, blockDim.x - 32);
    if (threadIdx.x == 0) {
        // release the CTA's phase writes (ordered before by the CTA barrier)
        // with the arrival itself; no returned value to wait for
        asm volatile("fence.proxy.async.global;" ::: "memory");
        asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(P.grid_bar) : "memory");
        // the next phase's tensor maps into the TMA descriptor cache meanwhile
        if (next_ph >= 0)
            for (int i = P.phase_prob[next_ph]; i < P.phase_prob[next_ph + 1]; ++i) {
                tma_prefetch_desc(&P.p[i].tmA);
                tma_prefetch_desc(&P.p[i].tmB);
                if (P.p[i].bulk_st || P.p[i].sym_tma) tma_prefetch_desc(&P.p[i].tmC);
            }
        const unsigned target = (unsigned)(seq + 1) * gridDim.x;
        uint64_t t0 = 0;
        while (true) {
            unsigned v;
            asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(P.grid_bar) : "memory");
            if (v >= target) break;
            if (t0 == 0) {
                t0 = globaltimer_ns();
            } else if (globaltimer_ns() - t0 > kWaitLimitNs) {
                *abort_flag = 1;
                set_status(P.status, MC_DEV_TIMEOUT);
                break;
            }
            __nanosleep(32);
        }
        asm volatile("fence.proxy.async.global;" ::: "memory");
    }
    __syncthreads();
    tc_fence_after();
}

MC_D void store_bf16x8(__nv_bfloat16* dst, const float* v) {
    __nv_bfloat162 h[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
    *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<uint4*>(h);
}
MC_D void store_f16x8(__half* dst, const float* v) {
    __half2 h[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2half2_rn(v[2 * i], v[2 * i + 1]);
    *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<uint4*>(h);
}

// The diagonal term: diag added to element (r, r) when the 32 x 64 chunk at
// (row0, col0) meets the diagonal (a warp-uniform test); the column is
// matched by an unrolled compare, so the values stay in registers.
MC_D void add_diag(const GemmProblem& q, int row0, int col0, int r, float* f) {
    if (q.diag == 0.f || col0 >= row0 + 32 || row0 >= col0 + 64) return;
    const float dg = q.diag;
#pragma unroll
    for (int i = 0; i < 64; ++i)
        if (col0 + i == r) f[i] = __fadd_rn(f[i], dg);
}

// Epilogue for 64 consecutive columns [col0, col0 + 64) of row r.
MC_D void epilogue_chunk(const GemmProblem& q, int z, int r, int col0, float* f, float sc, unsigned* status) {
    if (r >= q.M || col0 >= q.N) return;
    if (q.rope_tab && (col0 % q.rope_period) == q.rope_start) {
        const float2* cs = q.rope_tab + (size_t)(r % q.rope_T) * 32;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            float2 t = cs[i];
            float lo = f[i], hi = f[i + 32];
            f[i] = lo * t.x - hi * t.y;
            f[i + 32] = hi * t.x + lo * t.y;
        }
    }
    if (q.aux) {
        const __nv_bfloat16* ap = q.aux + (size_t)z * q.aux_bstride + (size_t)r * q.aux_ld + col0;
#pragma unroll
        for (int v = 0; v < 8; ++v) {
            uint4 u = *reinterpret_cast<const uint4*>(ap + 8 * v);
            const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
            const __half2* hf = reinterpret_cast<const __half2*>(&u);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 a2 = q.ab_f16 ? __half22float2(hf[i]) : __bfloat1622float2(h[i]);
                f[8 * v + 2 * i] = sc * (q.alpha * f[8 * v + 2 * i] + q.beta * a2.x);
                f[8 * v + 2 * i + 1] = sc * (q.alpha * f[8 * v + 2 * i + 1] + q.beta * a2.y);
            }
        }
    } else if (q.alpha != 1.0f || sc != 1.0f) {
        float s = sc * q.alpha;
#pragma unroll
        for (int i = 0; i < 64; ++i) f[i] *= s;
    }
    add_diag(q, r - (threadIdx.x & 31), col0, r, f);
    if (q.out_kind == kOutF16) {
        __half* o = reinterpret_cast<__half*>(q.out) + (size_t)z * q.out_bstride + (size_t)r * q.out_ld;
        bool big = false;
#pragma unroll
        for (int i = 0; i < 64; ++i) big |= fabsf(f[i]) > 65504.0f;
        if (big) set_status(status, MC_DEV_RANGE);
        if (q.vec_ok && col0 + 64 <= q.N) {
#pragma unroll
            for (int v = 0; v < 8; ++v) store_f16x8(o + col0 + 8 * v, f + 8 * v);
        } else {
#pragma unroll
            for (int i = 0; i < 64; ++i)
                if (col0 + i < q.N) o[col0 + i] = __float2half_rn(f[i]);
        }
        return;
    }
    if (q.out_kind == kOutF32) {
        float* o = reinterpret_cast<float*>(q.out) + (size_t)z * q.out_bstride + (size_t)r * q.out_ld;
        if (q.vec_ok && col0 + 64 <= q.N) {
#pragma unroll
            for (int v = 0; v < 16; ++v)
                *reinterpret_cast<float4*>(o + col0 + 4 * v) =
                    make_float4(f[4 * v], f[4 * v + 1], f[4 * v + 2], f[4 * v + 3]);
        } else {
#pragma unroll
            for (int i = 0; i < 64; ++i)
                if (col0 + i < q.N) o[col0 + i] = f[i];
        }
        return;
    }
    __nv_bfloat16* ob = reinterpret_cast<__nv_bfloat16*>(q.out) + (size_t)z * q.out_bstride;
    if (!q.sym) {
        __nv_bfloat16* o = ob + (size_t)r * q.out_ld;
        if (q.vec_ok && col0 + 64 <= q.N) {
#pragma unroll
            for (int v = 0; v < 8; ++v) store_bf16x8(o + col0 + 8 * v, f + 8 * v);
        } else {
#pragma unroll
            for (int i = 0; i < 64; ++i)
                if (col0 + i < q.N) o[col0 + i] = __float2bfloat16_rn(f[i]);
        }
        return;
    }
    // symmetric: keep c >= r, mirror to (c, r).  Lanes hold consecutive rows,
    // so the mirrored stores of one column are coalesced across the warp.
    if (q.vec_ok && col0 >= r && col0 + 64 <= q.N) {
        __nv_bfloat16* o = ob + (size_t)r * q.out_ld;
#pragma unroll
        for (int v = 0; v < 8; ++v) store_bf16x8(o + col0 + 8 * v, f + 8 * v);
#pragma unroll
        for (int i = 0; i < 64; ++i)
            ob[(size_t)(col0 + i) * q.out_ld + r] = __float2bfloat16_rn(f[i]);
    } else {
#pragma unroll
        for (int i = 0; i < 64; ++i) {
            int c = col0 + i;
            if (c >= r && c < q.N) {
                __nv_bfloat16 h = __float2bfloat16_rn(f[i]);
                ob[(size_t)r * q.out_ld + c] = h;
                ob[(size_t)c * q.out_ld + r] = h;
            }
        }
    }
}

MC_D uint4 pack8(const float* v, bool f16) {
    uint4 u;
    if (f16) {
        __half2* h = reinterpret_cast<__half2*>(&u);
#pragma unroll
        for (int i = 0; i < 4; ++i) h[i] = __floats2half2_rn(v[2 * i], v[2 * i + 1]);
    } else {
        __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
        for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
    }
    return u;
}

// Aux rows of a 32-row x 64-column chunk, one 16-byte segment per lane and
// pass (4 rows x 8 segments per pass): coalesced, issued early so that the
// loads are in flight while the accumulator is still being produced.
MC_D void aux_load(const GemmProblem& q, int z, int row0, int col0, uint4 (&u)[8]) {
    const int lane = threadIdx.x & 31;
    const int seg = lane & 7, sub = lane >> 3;
    const __nv_bfloat16* ab = q.aux + (size_t)z * q.aux_bstride + col0 + seg * 8;
#pragma unroll
    for (int it = 0; it < 8; ++it) {
        const int grow = row0 + it * 4 + sub;
        u[it] = (grow < q.M && col0 + seg * 8 < q.N) ? *reinterpret_cast<const uint4*>(ab + (size_t)grow * q.aux_ld)
                                                     : make_uint4(0, 0, 0, 0);
    }
}

// The chunk's values: RoPE, then v = sc (alpha acc + beta aux) with the aux
// segments u (from aux_load) transposed to one row per lane through the
// warp's staging buffer S.
MC_D void chunk_values(const GemmProblem& q, int row0, int col0, float* f, float sc, uint16_t* S,
                       const uint4 (&u)[8], bool swz) {
    const int lane = threadIdx.x & 31;
    const int r = row0 + lane;
    const int seg = lane & 7, sub = lane >> 3;
    if (q.rope_tab && (col0 % q.rope_period) == q.rope_start && r < q.M) {
        const float2* cs = q.rope_tab + (size_t)(r % q.rope_T) * 32;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            float2 t = cs[i];
            float lo = f[i], hi = f[i + 32];
            f[i] = lo * t.x - hi * t.y;
            f[i + 32] = hi * t.x + lo * t.y;
        }
    }
    if (q.aux) {
        // the problem's fields live in shared memory: read before the stores
        // to S, which the compiler must assume may alias them
        const bool aux_f16 = q.ab_f16 != 0;
        const float alpha = q.alpha, beta = q.beta;
#pragma unroll
        for (int it = 0; it < 8; ++it) *reinterpret_cast<uint4*>(S + stage_off(swz, it * 4 + sub, seg)) = u[it];
        __syncwarp();
        // v = sc (alpha acc + beta aux), pairs of values through the packed
        // fp32 arithmetic of sm_100+: beta aux, then one fused multiply-add,
        // then the scale, each rounded once
        const float2 al2 = make_float2(alpha, alpha), be2 = make_float2(beta, beta), sc2 = make_float2(sc, sc);
#pragma unroll
        for (int v = 0; v < 8; ++v) {
            uint4 w = *reinterpret_cast<const uint4*>(S + stage_off(swz, lane, v));
            const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&w);
            const __half2* hf = reinterpret_cast<const __half2*>(&w);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                // aux has the operands' type (fp16 or bf16)
                const float2 a2 = aux_f16 ? __half22float2(hf[i]) : __bfloat1622float2(h[i]);
                const float2 acc = make_float2(f[8 * v + 2 * i], f[8 * v + 2 * i + 1]);
                const float2 r = __fmul2_rn(sc2, __ffma2_rn(al2, acc, __fmul2_rn(be2, a2)));
                f[8 * v + 2 * i] = r.x;
                f[8 * v + 2 * i + 1] = r.y;
            }
        }
        __syncwarp();
    } else if (q.alpha != 1.0f || sc != 1.0f) {
        const float s = sc * q.alpha;
        const float2 s2 = make_float2(s, s);
#pragma unroll
        for (int i = 0; i < 64; i += 2) {
            const float2 r = __fmul2_rn(s2, make_float2(f[i], f[i + 1]));
            f[i] = r.x;
            f[i + 1] = r.y;
        }
    }
    add_diag(q, row0, col0, r, f);
}

// Warp-cooperative epilogue of a 32-row x 64-column chunk (rows row0.., one
// per lane; 16-bit output with vec_ok).  The results are staged in the
// warp's buffer S and written either by one TMA tensor store of the whole
// chunk (bulk_st: one request instead of one per row or segment, which is
// what limits the write rate of a few warps) or by coalesced 16-byte
// stores: the rows, and for symmetric
// outputs the mirrored rows (c, r) of every c >= r, where only the 16-byte
// segment that straddles the diagonal is written element-wise.  With
// next_col0 >= 0 the next chunk's aux rows are loaded into u once this
// chunk's are consumed.
MC_D void epilogue_chunk_staged(const GemmProblem& q, int z, int row0, int col0, float* f, float sc,
                                uint16_t* S, unsigned* status, uint4 (&u)[8], int next_col0,
                                const CUtensorMap* tmC) {
    const int lane = threadIdx.x & 31;
    if (col0 >= q.N) return;  // warp-uniform
    bulk_wait_read();  // this lane's bulk copies out of S (if any) have read it
    __syncwarp();      // every lane is done with the previous chunk's S
    const int seg = lane & 7, sub = lane >> 3;
    chunk_values(q, row0, col0, f, sc, S, u, q.bulk_st != 0);
    if (q.aux && next_col0 >= 0 && next_col0 < q.N) aux_load(q, z, row0, next_col0, u);
    const bool f16 = q.out_kind == kOutF16;
    if (f16) {
        // the largest magnitude against the fp16 range (NaN is not a range error)
        float mx = 0.f;
#pragma unroll
        for (int i = 0; i < 64; i += 2) mx = fmaxf(mx, fmaxf(fabsf(f[i]), fabsf(f[i + 1])));
        if (mx > 65504.0f) set_status(status, MC_DEV_RANGE);
    }
    if (q.bulk_st) {
        // the 32 x 64 box in the swizzled layout of the tensor store (each
        // lane rewrites only the segments of its own row that it read)
#pragma unroll
        for (int v = 0; v < 8; ++v) *reinterpret_cast<uint4*>(S + stage_off(true, lane, v)) = pack8(f + 8 * v, f16);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            tma_store_3d(tmC, S, col0, row0, z);
            bulk_commit();
        }
        return;
    }
#pragma unroll
    for (int v = 0; v < 8; ++v) *reinterpret_cast<uint4*>(S + lane * kStageLd + v * 8) = pack8(f + 8 * v, f16);
    uint16_t* ob = reinterpret_cast<uint16_t*>(q.out) + (size_t)z * q.out_bstride;
    __syncwarp();
    // rows: 8 passes of 4 rows x 8 segments
#pragma unroll
    for (int it = 0; it < 8; ++it) {
        const int rr = it * 4 + sub, grow = row0 + rr, c = col0 + seg * 8;
        if (grow >= q.M || c >= q.N) continue;
        const uint4 u = *reinterpret_cast<const uint4*>(S + rr * kStageLd + seg * 8);
        uint16_t* dst = ob + (size_t)grow * q.out_ld + c;
        if (!q.sym || c >= grow) {
            *reinterpret_cast<uint4*>(dst) = u;
        } else if (c + 7 >= grow) {
            const uint16_t* e = reinterpret_cast<const uint16_t*>(&u);
#pragma unroll
            for (int i = 0; i < 8; ++i)
                if (c + i >= grow) dst[i] = e[i];
        }
    }
    if (!q.sym) return;
    // mirror: output row c (col0 <= c < col0 + 64) gets columns row0..row0+31,
    // 8 per lane (4 lanes per row, 8 rows per pass)
#pragma unroll
    for (int it = 0; it < 8; ++it) {
        const int cc = it * 8 + (lane >> 2), rs = (lane & 3) * 8;
        const int c = col0 + cc, r0 = row0 + rs;
        if (c >= q.N || r0 >= q.M || c < r0) continue;  // all 8 have c < r: the row pass wrote them
        uint16_t e[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) e[i] = S[(rs + i) * kStageLd + cc];
        uint16_t* dst = ob + (size_t)c * q.out_ld + r0;
        if (c >= r0 + 7) {
            uint4 u;
            uint16_t* pu = reinterpret_cast<uint16_t*>(&u);
#pragma unroll
            for (int i = 0; i < 8; ++i) pu[i] = e[i];
            *reinterpret_cast<uint4*>(dst) = u;
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i)
                if (r0 + i <= c) dst[i] = e[i];
        }
    }
}

// The two warps whose rows form one 64-row half of the tile meet here:
// lane 0 of each arrives, every lane waits (bounded).  false (in every
// lane) when the wait gave up.
MC_D bool pair_sync(uint64_t* bar, uint32_t& ph, volatile int* abort_flag, unsigned* status) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
    const bool ok = mbar_wait(bar, ph, abort_flag, status);
    ph ^= 1;
    return ok;
}

// Symmetric 16-bit output, a 32 x 64 chunk wholly above the diagonal of its
// pair of warps (every column right of the pair's 64 rows): the rows go out
// as one TMA tensor store of the chunk, and the mirrored rows as two more.
// The pair transposes its 64 x 64 region into two {64, 32} boxes, rows
// c0 .. c0 + 31 in the buffer of the warp with the lower rows (S when low)
// and rows c0 + 32 .. c0 + 63 in the other's (Sp), each warp writing its 32
// columns of both; each warp then stores the box in its own buffer.  Four
// epilogue warps issue one global request per 128-byte row segment at about
// one per 15 cycles per SM; three TMA stores replace the 512 requests of the
// coalesced row and mirror stores.  The values are rounded once: the mirror
// holds the same 16-bit values as the rows.
MC_D bool epilogue_chunk_sym_tma(const GemmProblem& q, int z, int row0, int col0, float* f, float sc,
                                 uint16_t* S, uint64_t* pairbar, uint32_t& pph, unsigned* status, uint4 (&u)[8],
                                 int next_col0, const CUtensorMap* tmC, volatile int* abort_flag) {
    const int lane = threadIdx.x & 31;
    // warps 2 / 3 and 4 / 5 pair up (rows 64-127 and 0-63 of the tile); the
    // even warp holds the lower 32 rows, and the buffers are adjacent
    const int warp = threadIdx.x >> 5;
    const bool low = (warp & 1) == 0;
    uint16_t* Sp = S + (low ? 1 : -1) * (kEpiWarpBytes / 2);
    uint64_t* pbar = pairbar + ((warp & 3) >> 1);
    bulk_wait_read();  // this warp's stores of the previous chunk have read S
    __syncwarp();
    chunk_values(q, row0, col0, f, sc, S, u, true);
    if (q.aux && next_col0 >= 0 && next_col0 < q.N) aux_load(q, z, row0, next_col0, u);
    const bool f16 = q.out_kind == kOutF16;
    if (f16) {
        float mx = 0.f;
#pragma unroll
        for (int i = 0; i < 64; i += 2) mx = fmaxf(mx, fmaxf(fabsf(f[i]), fabsf(f[i + 1])));
        if (mx > 65504.0f) set_status(status, MC_DEV_RANGE);
    }
    // the 16-bit values, rounded once for the rows and the mirror
    uint4 pk[8];
#pragma unroll
    for (int v = 0; v < 8; ++v) pk[v] = pack8(f + 8 * v, f16);
    // both warps are past their aux staging in S and their previous stores
    // out of it: each warp's buffer is free for its own rows
    if (!pair_sync(pbar, pph, abort_flag, status)) return false;
#pragma unroll
    for (int v = 0; v < 8; ++v) *reinterpret_cast<uint4*>(S + stage_off(true, lane, v)) = pk[v];
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
        tma_store_3d(tmC, S, col0, row0, z);
        bulk_commit();
    }
    bulk_wait_read();  // the rows have been read out of S
    __syncwarp();
    // both buffers are free: the transposed halves go into both
    if (!pair_sync(pbar, pph, abort_flag, status)) return false;
    const int e = lane + (low ? 0 : 32);  // this row's column in the transposed boxes
    const int seg = e >> 3, el = e & 7;
    uint16_t* bA = low ? S : Sp;  // transposed rows c0 .. c0 + 31
    uint16_t* bB = low ? Sp : S;  // transposed rows c0 + 32 .. c0 + 63
#pragma unroll
    for (int v = 0; v < 8; ++v) {
        uint16_t* b = v < 4 ? bA : bB;
        const uint32_t w[4] = {pk[v].x, pk[v].y, pk[v].z, pk[v].w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int i = (v & 3) * 8 + 2 * k;  // row of the transposed box
            b[stage_off(true, i, seg) + el] = (uint16_t)(w[k] & 0xFFFFu);
            b[stage_off(true, i + 1, seg) + el] = (uint16_t)(w[k] >> 16);
        }
    }
    fence_proxy_async_smem();
    // the other warp's half of this warp's box is written and fenced
    if (!pair_sync(pbar, pph, abort_flag, status)) return false;
    if (lane == 0) {
        tma_store_3d(tmC, S, row0 - (low ? 0 : 32), col0 + (low ? 0 : 32), z);
        bulk_commit();
    }
    __syncwarp();
    return true;
}

// Pre-phase of a multi-phase Newton-Schulz launch: s = 1 / (||U||_F + eps)
// and s^2 from the momentum pass's per-tile sums of squares, one matrix per
// CTA at a time, summed in a fixed order.
template <int MAXP>
MC_D void norm_prephase(const GemmParamsT<MAXP>& P, double* red) {
    for (int z = P.norm_begin + blockIdx.x; z < P.norm_end; z += gridDim.x) {
        const MatInfo& mi = P.mats[z];
        double acc = 0.0;
        for (int i = threadIdx.x; i < mi.nparts; i += blockDim.x) acc += mi.partial[i];
        red[threadIdx.x] = acc;
        __syncthreads();
        if (threadIdx.x == 0) {
            double tot = 0.0;
            for (int i = 0; i < (int)blockDim.x; ++i) tot += red[i];
            const double den = sqrt(tot) + (double)P.eps;
            P.s[z] = (float)(1.0 / den);
            P.s2[z] = (float)(1.0 / (den * den));
        }
        __syncthreads();
    }
}

template <int MAXP, int BN, int STAGES, bool PAIR, int KS>
__global__ void __launch_bounds__(kGemmThreads, 1) gemm_kernel(const __grid_constant__ GemmParamsT<MAXP> P) {
    using Cfg = TileCfg<BN, STAGES, PAIR, KS>;
    constexpr int kKChunks = Cfg::kKChunks;
    constexpr int kAStageBytes = Cfg::kAStageBytes;
    constexpr int TM = Cfg::kTileM;
    constexpr int kBStageBytes = Cfg::kBStage;
    constexpr int kGemmStages = STAGES;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = smem;
    uint8_t* sB = smem + kGemmStages * kAStageBytes;
    uint16_t* sEpi = reinterpret_cast<uint16_t*>(sB + kGemmStages * kBStageBytes);
    auto* tail = reinterpret_cast<GemmSmemTail<STAGES>*>(sB + kGemmStages * kBStageBytes + 4 * kEpiWarpBytes);
    static_assert(sizeof(GemmSmemTail<STAGES>) <= kTailBytes, "tail");
    GemmProblem* sProb = reinterpret_cast<GemmProblem*>(
        (reinterpret_cast<uintptr_t>(tail) + kTailBytes + 63) & ~uintptr_t(63));
    volatile int* abort_flag = &tail->abort_flag;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // pair mode: cluster of two CTAs; rank 0 issues the MMAs of the pair
    const uint32_t rank = PAIR ? cluster_ctarank() : 0;
    const bool leader = rank == 0;
    const int unit = PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
    const int nunits = PAIR ? (int)(gridDim.x >> 1) : (int)gridDim.x;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kGemmStages; ++s) {
            mbar_init(&tail->full[s], 1);
            mbar_init(&tail->empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&tail->tfull[a], 1);
            mbar_init(&tail->tempty[a], PAIR ? 8 : 4);  // pair: both CTAs' epilogue warps
        }
        mbar_init(&tail->drain, 1);
        for (int pr = 0; pr < 2; ++pr) mbar_init(&tail->pairbar[pr], 2);  // lane 0 of both warps
        tail->abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        for (int i = 0; i < P.nprob; ++i) {
            tma_prefetch_desc(&P.p[i].tmA);
            tma_prefetch_desc(&P.p[i].tmB);
            if (P.p[i].bulk_st || P.p[i].sym_tma) tma_prefetch_desc(&P.p[i].tmC);
        }
    }
    if (warp == 1) {
        if constexpr (PAIR) {
            tmem_alloc_pair(&tail->tmem_base, Cfg::kTmemCols);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(&tail->tmem_base, Cfg::kTmemCols);
            tmem_relinquish();
        }
    }
    if (warp >= 2) stage_phase(P, 0, sProb, threadIdx.x - 64, blockDim.x - 64);
    tc_fence_before();
    __syncthreads();
    if constexpr (PAIR) cluster_sync();  // both CTAs' barriers and TMEM exist before any remote use
    tc_fence_after();
    const uint32_t tmem_base = tail->tmem_base;
    pdl_wait();  // the previous kernel's outputs are our inputs

    // role state, carried across phases
    int stage = 0, acc = 0;
    uint32_t phase = 0, aphase = 0;
    uint32_t pph = 0;  // epilogue warps: phase of their pair's barrier
    uint32_t issued[STAGES];
#pragma unroll
    for (int s = 0; s < STAGES; ++s) issued[s] = 0;
    bool ok = true;
    int nsync = 0;
    if (P.norm_end > P.norm_begin) {
        norm_prephase(P, reinterpret_cast<double*>(sEpi));
        grid_sync(P, nsync++, abort_flag, -1, nullptr);
    }

    for (int ph = 0; ph < P.nphase; ++ph) {
        const int pb = P.phase_prob[ph], np = P.phase_prob[ph + 1] - pb;
        const GemmProblem* sp = sProb + (ph & 1) * kPhaseProbs;
        const int t_begin = sp[0].tile_begin;
        const int t_end = sp[0].a_shared ? sp[0].tiles_m * (sp[np - 1].tn_off + sp[np - 1].tiles_n)
                                         : sp[np - 1].tile_begin + sp[np - 1].tiles_per_batch * sp[np - 1].batch;
        ok = ok && !*abort_flag;
        if (warp == 0 || warp == 6) {
            // ---------------- TMA producers ----------------
            // both walk every stage; warp 0 loads the A half (and arms the
            // full barrier with the whole stage's bytes), warp 6 the B half.
            // B bytes may land before the barrier is armed: the phase cannot
            // complete before warp 0's arrival, and the transaction count
            // only has to balance by then.
            const bool loads_a = warp == 0;
            if (lane == 0 && ok) {
                for (int t = t_begin + unit; t < t_end && ok; t += nunits) {
                    int pi, z, tm, tn;
                    decode_tile<BN, TM>(sp, np, t, pi, z, tm, tn);
                    const GemmProblem& q = sp[pi];
                    const CUtensorMap* tmA = &P.p[pb + pi].tmA;
                    const CUtensorMap* tmB = &P.p[pb + pi].tmB;
                    const int b_mn = q.b_mn;
                    const int nk = (q.K + KS - 1) / KS;
                    for (int kb = 0; kb < nk; ++kb) {
                        if (!mbar_wait(&tail->empty[stage], phase ^ 1, abort_flag, P.status)) {
                            ok = false;
                            break;
                        }
                        uint8_t* a = sA + stage * kAStageBytes;
                        uint8_t* b = sB + stage * kBStageBytes;
                        const int k0 = kb * KS;
                        if constexpr (PAIR) {
                            // both CTAs' halves complete on the leader's full barrier
                            const uint32_t fb = mapa_shared(smem_u32(&tail->full[stage]), 0);
                            if (loads_a) {
                                if (leader)
                                    mbar_arrive_expect_tx(&tail->full[stage], 2 * (kAStageBytes + kBStageBytes));
#pragma unroll
                                for (int c = 0; c < kKChunks; ++c)
                                    tma_load_3d_pair(a + c * kAChunkBytes, tmA, fb, k0 + c * kBK,
                                                     tm * TM + rank * kBM, z);
                            } else {
                                const int b0 = tn * BN + (int)rank * Cfg::kBRows;
                                if (!b_mn) {
#pragma unroll
                                    for (int c = 0; c < kKChunks; ++c)
                                        tma_load_3d_pair(b + c * Cfg::kBChunkK, tmB, fb, k0 + c * kBK, b0, z);
                                } else {
#pragma unroll
                                    for (int j = 0; j < Cfg::kBRows / 64; ++j)
                                        tma_load_3d_pair(b + j * Cfg::kBChunkMN, tmB, fb, b0 + j * 64, k0, z);
                                }
                            }
                        } else {
                            if (loads_a) {
                                mbar_arrive_expect_tx(&tail->full[stage], kAStageBytes + kBStageBytes);
#pragma unroll
                                for (int c = 0; c < kKChunks; ++c)
                                    tma_load_3d(a + c * kAChunkBytes, tmA, &tail->full[stage], k0 + c * kBK, tm * kBM, z);
                            } else if (!b_mn) {
#pragma unroll
                                for (int c = 0; c < kKChunks; ++c)
                                    tma_load_3d(b + c * Cfg::kBChunkK, tmB, &tail->full[stage], k0 + c * kBK, tn * BN, z);
                            } else {
#pragma unroll
                                for (int j = 0; j < BN / 64; ++j)
                                    tma_load_3d(b + j * Cfg::kBChunkMN, tmB, &tail->full[stage], tn * BN + j * 64, k0, z);
                            }
                        }
                        ++issued[stage];
                        if (++stage == kGemmStages) {
                            stage = 0;
                            phase ^= 1;
                        }
                    }
                }
            }
        } else if (warp == 1) {
            // ---------------- MMA issuer (the leader of a pair) ----------------
            for (int t = t_begin + unit; t < t_end && ok && leader; t += nunits) {
                int pi, z, tm, tn;
                decode_tile<BN, TM>(sp, np, t, pi, z, tm, tn);
                const GemmProblem& q = sp[pi];
                const int nk = (q.K + KS - 1) / KS;
                const int b_mn = q.b_mn;
                const uint32_t idesc = idesc_f16kind(TM, BN, b_mn, q.ab_f16);
                if (!mbar_wait(&tail->tempty[acc], aphase ^ 1, abort_flag, P.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
                for (int kb = 0; kb < nk; ++kb) {
                    if (!mbar_wait(&tail->full[stage], phase, abort_flag, P.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    if (lane == 0) {
                        // stage descriptors once; a K step moves the 16-byte
                        // address field: +32 B within a K-major chunk, +16 KB
                        // (A) or one B chunk to the next chunk, +2 KB per
                        // step down an MN-major chunk
                        const uint64_t a_d = sw128_desc(smem_u32(sA + stage * kAStageBytes), 16, 1024);
                        const uint64_t b_d = b_mn ? sw128_desc(smem_u32(sB + stage * kBStageBytes), Cfg::kBChunkMN, 1024)
                                                  : sw128_desc(smem_u32(sB + stage * kBStageBytes), 16, 1024);
#pragma unroll
                        for (int k = 0; k < KS / 16; ++k) {
                            const uint64_t ad = a_d + (uint64_t)((k >> 2) * (kAChunkBytes >> 4) + (k & 3) * 2);
                            const uint64_t bd = b_mn ? b_d + (uint64_t)(k * (2048 >> 4))
                                                     : b_d + (uint64_t)((k >> 2) * (Cfg::kBChunkK >> 4) + (k & 3) * 2);
                            if constexpr (PAIR)
                                umma_pair(d_tmem, ad, bd, idesc, (kb | k) != 0);
                            else
                                umma_bf16(d_tmem, ad, bd, idesc, (kb | k) != 0);
                        }
                        if constexpr (PAIR)
                            umma_commit_pair_both(&tail->empty[stage]);  // both producers may refill
                        else
                            umma_commit(&tail->empty[stage]);
                    }
                    __syncwarp();
                    if (++stage == kGemmStages) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
                if (!ok) break;
                if (lane == 0) {
                    if constexpr (PAIR)
                        umma_commit_pair_both(&tail->tfull[acc]);  // both epilogues
                    else
                        umma_commit(&tail->tfull[acc]);
                }
                __syncwarp();
                if (++acc == 2) {
                    acc = 0;
                    aphase ^= 1;
                }
            }
        } else if (warp <= 5) {
            // ---------------- epilogue (warps 2..5) ----------------
            const int quarter = warp & 3;  // TMEM lanes this warp may access
            uint16_t* S = sEpi + (warp - 2) * (kEpiWarpBytes / 2);
            for (int t = t_begin + unit; t < t_end && ok; t += nunits) {
                int pi, z, tm, tn;
                decode_tile<BN, TM>(sp, np, t, pi, z, tm, tn);
                const GemmProblem& q = sp[pi];
                const bool staged = q.vec_ok && q.out_kind != kOutF32;
                const int row0 = tm * TM + (int)rank * kBM + quarter * 32;
                uint4 u[8] = {};
                if (staged && q.aux) aux_load(q, z, row0, tn * BN, u);
                if (!mbar_wait(&tail->tfull[acc], aphase, abort_flag, P.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const int r = row0 + lane;
                const float sc = q.scale ? q.scale[z] : 1.0f;
#pragma unroll 1
                for (int c = 0; c < BN / 64; ++c) {
                    uint32_t v[64];
                    uint32_t taddr = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * BN + c * 64);
                    tmem_ld32(taddr, v);
                    tmem_ld32(taddr + 32, v + 32);
                    tmem_ld_wait();
                    const int col0 = tn * BN + c * 64;
                    const int pair_row0 = row0 & ~63;  // the pair's 64 rows (row blocks are multiples of 64)
                    // CTA-pair tiles only: the single-CTA launches of small
                    // batches keep the compact epilogue
                    if (PAIR && staged && q.sym_tma && col0 >= pair_row0 + 64 && pair_row0 + 64 <= q.M &&
                        col0 + 64 <= q.N) {
                        if (!epilogue_chunk_sym_tma(q, z, row0, col0, reinterpret_cast<float*>(v), sc, S,
                                                    tail->pairbar, pph, P.status, u,
                                                    c + 1 < BN / 64 ? tn * BN + (c + 1) * 64 : -1,
                                                    &P.p[pb + pi].tmC, abort_flag)) {
                            ok = false;
                            break;
                        }
                    } else if (staged)
                        epilogue_chunk_staged(q, z, row0, tn * BN + c * 64, reinterpret_cast<float*>(v), sc, S,
                                              P.status, u, c + 1 < BN / 64 ? tn * BN + (c + 1) * 64 : -1,
                                              &P.p[pb + pi].tmC);
                    else
                        epilogue_chunk(q, z, r, tn * BN + c * 64, reinterpret_cast<float*>(v), sc, P.status);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    if (PAIR && !leader)
                        mbar_arrive_cluster(mapa_shared(smem_u32(&tail->tempty[acc]), 0));
                    else
                        mbar_arrive(&tail->tempty[acc]);
                }
                if (++acc == 2) {
                    acc = 0;
                    aphase ^= 1;
                }
            }
            // this lane's bulk copies are written before the phase ends
            bulk_wait_all();
            asm volatile("fence.proxy.async.global;" ::: "memory");
        }
        if (ph + 1 < P.nphase) grid_sync(P, nsync++, abort_flag, ph + 1, sProb + ((ph + 1) & 1) * kPhaseProbs);
    }

    if ((warp == 0 || warp == 6) && lane == 0 && leader) {
        // wait for the copies still in flight before exit (a pair's copies all
        // complete on the leader's barriers; the final cluster barrier keeps
        // the other CTA resident until then)
        volatile int never = 0;
        for (int s = 0; s < kGemmStages; ++s)
            if (issued[s]) mbar_wait(&tail->full[s], (issued[s] - 1) & 1, &never, P.status);
    } else if (warp == 1 && leader) {
        // drain: every MMA this thread issued has completed before teardown
        if (lane == 0) {
            if constexpr (PAIR)
                umma_commit_pair(&tail->drain);
            else
                umma_commit(&tail->drain);
        }
        __syncwarp();
        volatile int never = 0;
        mbar_wait(&tail->drain, 0, &never, P.status);
    }

    pdl_trigger();
    tc_fence_before();
    __syncthreads();
    if constexpr (PAIR) cluster_sync();  // the leader's MMAs and remote arrivals are done
    tc_fence_after();
    if (warp == 1) {
        if constexpr (PAIR)
            tmem_dealloc_pair(tmem_base, Cfg::kTmemCols);
        else
            tmem_dealloc(tmem_base, Cfg::kTmemCols);
    }
}

template <int MAXP, int BN, int STAGES, bool PAIR, int KS>
static cudaError_t set_smem_attr() {
    static bool attr_set[64] = {false};
    int dev = current_device();
    if (dev < 0) return cudaErrorInvalidDevice;
    if (dev < 64 && !attr_set[dev]) {
        cudaError_t e = cudaFuncSetAttribute(gemm_kernel<MAXP, BN, STAGES, PAIR, KS>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             TileCfg<BN, STAGES, PAIR, KS>::kSmem);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    return cudaSuccess;
}

static_assert(sizeof(GemmParamsMulti) <= 32764, "kernel parameters");
// every phase holds 1..kPhaseProbs problems (the shared-memory staging size)
template <int MAXP>
static bool phases_fit(const GemmParamsT<MAXP>& P) {
    if (P.nphase < 1 || P.nphase > kMaxPhases) return false;
    for (int ph = 0; ph < P.nphase; ++ph) {
        const int n = P.phase_prob[ph + 1] - P.phase_prob[ph];
        if (n < 1 || n > kPhaseProbs) return false;
    }
    return P.phase_prob[P.nphase] == P.nprob;
}

// One persistent CTA (pair: one cluster of two CTAs) per SM (pair of SMs),
// no more than there are tiles; cooperative launches keep every CTA resident
// for the grid barriers between phases.
template <int MAXP, int BN, int STAGES, bool PAIR, int KS>
static cudaError_t launch_cfg(const GemmParamsT<MAXP>& P, bool coop, cudaStream_t stream, const char* label) {
    using Cfg = TileCfg<BN, STAGES, PAIR, KS>;
    static_assert(Cfg::kSmem <= 232448, "shared memory");
    if (P.tile_m != Cfg::kTileM || P.bn != BN) return cudaErrorInvalidValue;
    cudaError_t e = set_smem_attr<MAXP, BN, STAGES, PAIR, KS>();
    if (e != cudaSuccess) return e;
    int units = PAIR ? num_sms() / 2 : num_sms();
    if (!coop && units > P.total_tiles) units = P.total_tiles;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(PAIR ? 2 * units : units);
    cfg.blockDim = dim3(kGemmThreads);
    cfg.dynamicSmemBytes = Cfg::kSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    int na = 0;
    if (coop) {
        attr[na].id = cudaLaunchAttributeCooperative;
        attr[na].val.cooperative = 1;
        ++na;
    } else {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    if (PAIR) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = 2;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    TraceScope ts(label, stream);
    e = cudaLaunchKernelEx(&cfg, gemm_kernel<MAXP, BN, STAGES, PAIR, KS>, P);
    return e != cudaSuccess ? e : cudaGetLastError();
}

// Configurations: 256 x 256 tiles on CTA pairs (projections, plain GEMMs,
// large Newton-Schulz batches) and 128 x 128 tiles on single CTAs (small
// Newton-Schulz batches), with the stage shapes of internal.h.
cudaError_t launch_gemm(const GemmParams& P, cudaStream_t stream, const char* label) {
    if (P.total_tiles <= 0) return cudaSuccess;
    if (!phases_fit(P)) return cudaErrorInvalidValue;
    return launch_cfg<kMaxProblems, kBN, kStagesPair, true, kStageKPair>(P, false, stream, label);
}

cudaError_t launch_gemm_multi(const GemmParamsMulti& P, cudaStream_t stream, const char* label) {
    if (P.total_tiles <= 0) return cudaSuccess;
    if (!phases_fit(P)) return cudaErrorInvalidValue;
    if (P.tile_m == 2 * kBM)
        return launch_cfg<kMaxProblemsMulti, kBN, kStagesPair, true, kStageKPair>(P, true, stream, label);
    return launch_cfg<kMaxProblemsMulti, 128, kStagesSingle, false, kStageKSingle>(P, true, stream, label);
}

}  // namespace mc
