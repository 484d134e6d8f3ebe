// internal.h -- host-side interfaces shared by the translation units of the
// library (not part of the public ABI).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/mc_max.h"

namespace mc {

// ---------------------------------------------------------------------------
// tile geometry of the tensor-core kernels
// ---------------------------------------------------------------------------
constexpr int kBM = 128;  // UMMA M (TMEM lanes)
constexpr int kBN = 256;  // UMMA N (TMEM columns per accumulator)
constexpr int kBK = 64;   // K of one 128-byte swizzle row of bf16: one TMA box, one descriptor chunk
// K per pipeline stage and ring depth of the two GEMM configurations: CTA
// pairs (256-wide tiles) and single CTAs (128 x 128 tiles).  A stage holds
// K / 64 swizzle chunks; its MMAs (K = 16 each) share one commit.
#ifndef MC_PAIR_STAGE_K
#define MC_PAIR_STAGE_K 128
#endif
#ifndef MC_PAIR_STAGES
#define MC_PAIR_STAGES 3
#endif
constexpr int kStageKPair = MC_PAIR_STAGE_K;
constexpr int kStagesPair = MC_PAIR_STAGES;
constexpr int kStageKSingle = 128;
constexpr int kStagesSingle = 3;
constexpr int stage_k_for(int tile_m) { return tile_m == 2 * kBM ? kStageKPair : kStageKSingle; }
constexpr int kMaxProblems = 4;        // problems of a single-phase launch
constexpr int kMaxProblemsMulti = 48;  // problems of a multi-phase launch (kernel parameters < 32 KB)
constexpr int kMaxPhases = 16;
constexpr int kPhaseProbs = 4;  // problems per phase (staged in shared memory)

// One GEMM problem of a multi-problem launch: D[z] = A[z] * op(B[z]),
// A [M][K] K-major; B K-major ([N][K]) or MN-major ([K][N]).
// Operands are bf16 or (ab_f16) fp16.  Epilogue: v = scale[z] * (alpha *
// acc + beta * aux[z][r][c]) (+ diag where r == c), optional RoPE on column
// chunks, then a bf16,
// f32 or f16 store (f16 stores flag MC_DEV_RANGE when |v| > 65504); `sym`
// stores only c >= r and mirrors it to (c, r) (M == N, only upper tiles are
// scheduled).
constexpr int kOutBF16 = 0, kOutF32 = 1, kOutF16 = 2;

struct GemmProblem {
    CUtensorMap tmA;  // 3D {K, M, batch}, box {64, 128}, 128B swizzle
    CUtensorMap tmB;  // K-major {K, N, batch} box {64, rows}; MN-major {N, K, batch} box {64, 128}
    CUtensorMap tmC;  // bulk_st: the 16-bit output {N, M, batch}, box {64, 32}, 128B swizzle
    int M, N, K, batch;
    int b_mn, sym, out_kind, vec_ok;  // out_kind: kOutBF16 / kOutF32 / kOutF16
    int ab_f16;
    int bulk_st;  // non-symmetric 16-bit output written by TMA tensor stores through tmC
    int a_shared; // the phase's problems share A: tiles go row block by row block across them
    int tn_off;   // a_shared: this problem's first column tile in the row block
    int tiles_m, tiles_n, tiles_per_batch, tile_begin;
    void* out;
    long long out_ld, out_bstride;
    const __nv_bfloat16* aux;
    long long aux_ld, aux_bstride;
    float alpha, beta;
    const float* scale;
    const float2* rope_tab;  // [rope_T][32] (cos, sin); null = no RoPE
    int rope_T, rope_period, rope_start;
    float diag;  // added to the diagonal elements (row == column) of the output, after alpha, beta and the scale
    int sym_tma;  // sym with a 16-bit output and tmC: chunks above the diagonal go out by TMA stores (rows and mirror)
    int pad_[3];
};
static_assert(sizeof(GemmProblem) % 16 == 0, "problems are staged in 16-byte pieces");

// Per-matrix facts of a Muon batch, written to the workspace by the
// momentum pass and read by the norm pre-phase of the multi-phase
// Newton-Schulz launch.
struct MatInfo {
    const double* partial;   // per-tile sums of squares of the Newton-Schulz input
    int nparts, pad_;
};

// A launch: problems in tile order.  With nphase > 1 the problems form
// consecutive phases (phase i = problems [phase_prob[i], phase_prob[i+1]));
// every CTA finishes its tiles of a phase before any CTA starts the next
// (grid barrier on *grid_bar, a zeroed counter; cooperative launch).
template <int MAXP>
struct GemmParamsT {
    GemmProblem p[MAXP];
    int nprob, total_tiles;
    int bn;      // output tile width of the launch: 256 (default when 0) or 128
    int tile_m;  // output tile height: 128 (one CTA, default when 0) or 256 (a CTA pair)
    int a_shared;  // single-phase launch whose problems share A (same rows, batch 1, not symmetric)
    int nphase;
    int phase_prob[kMaxPhases + 1];
    unsigned* grid_bar;
    unsigned* status;
    // multi-phase Newton-Schulz extras
    const MatInfo* mats;
    int norm_begin, norm_end;  // pre-phase: s, s2 of matrices [norm_begin, norm_end)
    float eps;
    float* s;
    float* s2;
};
using GemmParams = GemmParamsT<kMaxProblems>;
using GemmParamsMulti = GemmParamsT<kMaxProblemsMulti>;

// ---------------------------------------------------------------------------
// helpers (abi.cu)
// ---------------------------------------------------------------------------
unsigned* device_status_ptr();  // per-device status word (static device storage)
int num_sms();
int current_device();

// Counts every launch and, when tracing is on, brackets it with events on
// the launching stream.  Construct right before a launch, destroy right after.
class TraceScope {
public:
    TraceScope(const char* name, cudaStream_t stream);
    ~TraceScope();
private:
    const char* name_;
    cudaStream_t stream_;
    cudaEvent_t start_;
};

// 3D tensor map of 2-byte elements (bf16, or fp16 when f16 != 0) with
// 128-byte swizzle: dims {inner, outer, batch}, strides in elements; box
// {box_inner, box_outer, 1}.  false on failure.
bool make_tmap_3d(CUtensorMap* tm, const void* base, uint64_t inner, uint64_t outer,
                  uint64_t batch, uint64_t outer_stride, uint64_t batch_stride,
                  uint32_t box_inner, uint32_t box_outer, int f16,
                  bool swizzle = true);

// Fills the tile bookkeeping of problems [0, nprob), total_tiles and (when
// nphase is 0) a single phase.
template <int MAXP>
void finalize_gemm_params(GemmParamsT<MAXP>& P);

// gemm.cu
cudaError_t launch_gemm(const GemmParams& P, cudaStream_t stream, const char* label);
cudaError_t launch_gemm_multi(const GemmParamsMulti& P, cudaStream_t stream, const char* label);

// scan.cu
struct ScanArgs {
    // Q storage [B][T][q_ld], K main storage [B][T][k_ld], k^R storage
    // [B][T][kr_ld] (MLA only, may be null); all fp16
    const void* q;
    long long q_ld;
    const void* k;
    long long k_ld;
    const void* kr;
    long long kr_ld;
    int B, T, H, causal;
    int q_head_stride;   // columns between heads in Q
    int k_head_stride;   // columns between heads in K main
    int nkb_main;        // 64-wide K blocks per head read from K main
    int nkb_rope;        // 0 or 1 block read from k^R at column kr_col
    int kr_col;
    float d;
    // S = max / sqrt(d) is max-merged into s_max[H] (and s_bh[B][H] when
    // given), which hold 0xFFFFFFFF in every word before the launch, or the
    // maxima the scan accumulates into
    float* s_max;
    float* s_bh;
};
cudaError_t launch_scan(const ScanArgs& a, cudaStream_t stream);

// Attention forward with the max logit taken along (attn.cu) -------------------
struct AttnArgs {
    const void* q;       // bf16 [B][T][H*dh]; MLA: [B][T][H*(nope+rope)], q^C then q^R per head
    const void* k;       // MLA: k^C [B][T][H*nope]
    const void* v;       // MLA: [B][T][H*dv]
    const void* kr;      // MLA only: the shared k^R, rows of kr_ld elements, rope columns from kr_col
    int kr_ld, kr_col;
    int mla;             // 1: MLA with nope = 128, rope = 64, dv = 128 (dh = 192 for the logits)
    void* o;             // bf16 [B][T][H*dh]; MLA: [B][T][H*dv]
    int B, T, H, dh, causal;
    // S = max / sqrt(dh) merged into s_max / s_bh as in the scan
    float* s_max;
    float* s_bh;
};
cudaError_t launch_attn(const AttnArgs& a, cudaStream_t stream);

// fp32 CUDA-core fallbacks for small or unaligned MHA shapes
cudaError_t launch_proj_simt(const void* x, const void* w, mc_dtype dt, float* out, int rows,
                             int D, int N, cudaStream_t stream);
cudaError_t launch_scan_simt(const float* q, const float* k, int B, int T, int H, int dh,
                             int causal, unsigned* keys, cudaStream_t stream);

// keys [B][H] -> s_max[H] (max over B), s_bh[B][H]; S = key / sqrt(d)
cudaError_t launch_finalize_smax(const unsigned* keys, int B, int H, float d, int accumulate,
                                 float* s_max, float* s_bh, cudaStream_t stream);

// RoPE table [T][32] of (cos, sin)(t * base^(-2f/64)) in float2
cudaError_t launch_rope_table(float2* tab, int T, float base, cudaStream_t stream);

// elementwise.cu -------------------------------------------------------------
// one column segment of one weight matrix that a head's clip factor scales
struct ClipSeg {
    void* w;
    long long ld;       // row length (elements)
    int rows;
    int col0;           // first column of head 0's segment
    int head_stride;    // columns between heads
    int width;          // columns per head segment
    int use_gamma;      // 1: x gamma, 0: x sqrt(gamma)
};
constexpr int kMaxClipSegs = 4;
struct ClipArgs {
    ClipSeg seg[kMaxClipSegs];
    int nseg, H, bf16;
    const float* s_max;
    float tau;
    float* gamma_out;
};
cudaError_t launch_clip(const ClipArgs& a, cudaStream_t stream);
// dst[i] = fp16(src[i]) for bf16 src (exact in fp16's normal range)
cudaError_t launch_bf16_to_f16(const void* src, void* dst, long long n, cudaStream_t stream);
cudaError_t launch_clip_global(void* wq, void* wk, int bf16, long long n, const float* s_max,
                               int H, float tau, float alpha, float* gamma_out,
                               cudaStream_t stream);

// Muon elementwise passes over a batch of matrices ---------------------------
constexpr int kMaxBatchMats = 32;  // per launch (kernel-parameter table, < 4 KB)
struct MatDesc {
    float* w;            // mode 2: weights [rows][cols] f32 (updated); mode 3: output O
    const float* g;      // mode 0: gradient [rows][cols]
    float* m;            // mode 0: momentum (updated); mode 1: the Newton-Schulz input
    __nv_bfloat16* x;    // [m_pad][n_pad] workspace in X orientation: bf16 (modes 0/1; modes 2/3
                         // with zero NS steps), fp16 (modes 2/3: the Newton-Schulz output)
    double* partial;     // modes 0/1: per-tile sums of squares
    const float* oscale; // modes 2/3: optional device scale of O (zero NS steps)
    float rms;           // mode 2: rms_coef * sqrt(max(rows, cols))
    int rows, cols, tr;  // tr: X = transpose of the matrix (rows > cols)
    int vec;             // cols % 4 == 0 and 16-byte aligned rows: float4 accesses
    int flat;            // X has the source's layout (vec, no transpose, no padding): 4096-element chunks
    int m_pad, n_pad;
    int tiles_x, tile_begin;  // 64 x 64 tiles over X [m_pad][n_pad]
};
struct MatBatch {
    MatDesc d[kMaxBatchMats];
    MatInfo* info;  // modes 0/1: info[info_base + i] is written for matrix i
    int info_base;
    int count, total_tiles;
    float mu, lr, wd;
    int nesterov, mode;  // 0 momentum + cast, 1 cast only, 2 update W, 3 write O
    int x_f16;           // modes 2/3: X holds fp16 (the Newton-Schulz output)
};
cudaError_t launch_mat_pass(const MatBatch& b, cudaStream_t stream);
// flat passes over one ZeRO-1 shard, and the S_max <-> int32 key maps
cudaError_t launch_momentum_flat(float* m, const float* g, float* u, long long n, float mu, float gs,
                                 int nesterov, cudaStream_t stream);
cudaError_t launch_update_flat(float* w, const float* o, long long n, float lr, float rms, float wd,
                               cudaStream_t stream);
cudaError_t launch_smax_keys(const float* s, int* keys, const int* kin, float* sout, int n, cudaStream_t stream);
// bounded-wait self-test (one CTA of two waiting warps; elementwise.cu)
cudaError_t launch_wait_selftest(uint64_t limit_ns, long long* out, cudaStream_t stream);

// s[z] = 1 / (sqrt(sum partial[z]) + eps), s2[z] = s[z]^2
struct NormArgs {
    const double* partial[kMaxBatchMats];
    int nparts[kMaxBatchMats];
    int count;
    float eps;
    float* s;
    float* s2;
};
cudaError_t launch_norm_finalize(const NormArgs& a, cudaStream_t stream);

}  // namespace mc
