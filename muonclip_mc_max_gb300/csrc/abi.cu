// abi.cu -- the C ABI of include/mc_max.h: argument checks, workspace
// carving, tensor-map encoding and launch sequencing on the caller's stream.
// Nothing here allocates device memory at run time; every buffer is the
// caller's.  The library's only device storage is static and part of its
// device module: the 4-byte status word and the 64 MiB scratch array of
// mc_max_logits_mha_noalloc.  The module is loaded on a device the first
// time any entry point runs there, so every device where the library has
// run holds both until the process exits.
#include <algorithm>
#include <atomic>
#include <map>
#include <mutex>
#include <string>
#include <vector>

#include "common.cuh"
#include "internal.h"

namespace mc {

// ---------------------------------------------------------------------------
// device helpers
// ---------------------------------------------------------------------------
__device__ unsigned g_status_word;  // per-device status bits (MC_DEV_*)

static std::mutex g_mu;
static std::mutex g_launch_mu;  // guards the static multi-phase parameter block
static unsigned* g_status_ptr[64];
static int g_sms[64];

int current_device() {
    int d = -1;
    if (cudaGetDevice(&d) != cudaSuccess) return -1;
    return d;
}

unsigned* device_status_ptr() {
    int dev = current_device();
    if (dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_status_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_status_word) == cudaSuccess) g_status_ptr[dev] = (unsigned*)p;
    }
    return g_status_ptr[dev];
}

int num_sms() {
    int dev = current_device();
    if (dev < 0 || dev >= 64) return 1;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_sms[dev]) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        g_sms[dev] = n > 0 ? n : 1;
    }
    return g_sms[dev];
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

bool make_tmap_3d(CUtensorMap* tm, const void* base, uint64_t inner, uint64_t outer, uint64_t batch,
                  uint64_t outer_stride, uint64_t batch_stride, uint32_t box_inner, uint32_t box_outer, int f16,
                  bool swizzle) {
    EncodeTiledFn fn = encode_fn();
    if (!fn || !base || (reinterpret_cast<uintptr_t>(base) & 15)) return false;
    if (batch == 1) batch_stride = outer_stride * outer;
    cuuint64_t dims[3] = {inner, outer, batch};
    cuuint64_t strides[2] = {outer_stride * 2, batch_stride * 2};
    if ((strides[0] & 15) || (strides[1] & 15)) return false;
    cuuint32_t box[3] = {box_inner, box_outer, 1};
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = fn(tm, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Projection and plain GEMM launches use 256-row tiles computed by CTA pairs
// (cta_group::2: each SM loads half of B).
constexpr int kPairTileM = 2 * kBM;

template <int MAXP>
void finalize_gemm_params(GemmParamsT<MAXP>& P) {
    int begin = 0;
    if (P.bn <= 0) P.bn = kBN;
    if (P.tile_m <= 0) P.tile_m = kBM;
    for (int i = 0; i < P.nprob; ++i) {
        GemmProblem& q = P.p[i];
        q.tiles_m = (q.M + P.tile_m - 1) / P.tile_m;
        q.tiles_n = (q.N + P.bn - 1) / P.bn;
        if (q.sym) {
            // row block tm keeps the column tiles that reach the diagonal
            int t = 0;
            for (int tm = 0; tm < q.tiles_m; ++tm) t += q.tiles_n - (P.tile_m * tm) / P.bn;
            q.tiles_per_batch = t;
        } else {
            q.tiles_per_batch = q.tiles_m * q.tiles_n;
        }
        q.tile_begin = begin;
        begin += q.tiles_per_batch * q.batch;
    }
    P.total_tiles = begin;
    // shared A (one phase, same rows, batch 1, not symmetric): every row
    // block's column tiles of all problems run together, so A is read once
    bool shared = P.a_shared && P.nphase <= 1 && P.nprob > 1;
    for (int i = 0; shared && i < P.nprob; ++i)
        shared = P.p[i].M == P.p[0].M && P.p[i].batch == 1 && !P.p[i].sym;
    int tn = 0;
    for (int i = 0; i < P.nprob; ++i) {
        GemmProblem& q = P.p[i];
        q.a_shared = shared ? 1 : 0;
        q.tn_off = shared ? tn : 0;
        tn += q.tiles_n;
        if (shared) q.tile_begin = 0;
    }
    P.a_shared = shared ? 1 : 0;
    P.status = device_status_ptr();
    if (P.nphase <= 0) {
        P.nphase = 1;
        P.phase_prob[0] = 0;
        P.phase_prob[1] = P.nprob;
    }
}
template void finalize_gemm_params<kMaxProblems>(GemmParamsT<kMaxProblems>&);
template void finalize_gemm_params<kMaxProblemsMulti>(GemmParamsT<kMaxProblemsMulti>&);

// ---------------------------------------------------------------------------
// launch counting and optional event tracing
// ---------------------------------------------------------------------------
static std::atomic<unsigned long long> g_launches{0};
static std::atomic<int> g_trace_on{0};
struct TraceRec {
    const char* name;
    cudaEvent_t a, b;
};
static std::mutex g_trace_mu;
static std::vector<TraceRec> g_trace;
static std::vector<cudaEvent_t> g_event_pool;

static cudaEvent_t pooled_event() {
    std::lock_guard<std::mutex> lk(g_trace_mu);
    if (!g_event_pool.empty()) {
        cudaEvent_t e = g_event_pool.back();
        g_event_pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    return e;
}

// During stream capture an event becomes a graph node (re-recorded on every
// replay) only when recorded as an external event.
static void record_event(cudaEvent_t e, cudaStream_t s) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    cudaStreamIsCapturing(s, &cs);
    if (cs == cudaStreamCaptureStatusActive) cudaEventRecordWithFlags(e, s, cudaEventRecordExternal);
    else cudaEventRecord(e, s);
}

TraceScope::TraceScope(const char* name, cudaStream_t stream) : name_(name), stream_(stream), start_(nullptr) {
    g_launches.fetch_add(1, std::memory_order_relaxed);
    if (g_trace_on.load(std::memory_order_relaxed)) {
        start_ = pooled_event();
        if (start_) record_event(start_, stream_);
    }
}

TraceScope::~TraceScope() {
    if (!start_) return;
    cudaEvent_t end = pooled_event();
    if (!end) return;
    record_event(end, stream_);
    std::lock_guard<std::mutex> lk(g_trace_mu);
    g_trace.push_back(TraceRec{name_, start_, end});
}

static size_t align256(size_t b) { return (b + 255) & ~size_t(255); }

// bump allocator over the caller's workspace
// a * b, or SIZE_MAX when the product does not fit size_t
static size_t mul_sat(size_t a, size_t b) { return (a && b > SIZE_MAX / a) ? SIZE_MAX : a * b; }
static size_t mul_sat(size_t a, size_t b, size_t c) { return mul_sat(mul_sat(a, b), c); }

// Carves 256-byte-aligned pieces out of a workspace (or, with base null,
// only sums their sizes).  The sum saturates at SIZE_MAX instead of
// wrapping, so a size that does not fit size_t can never pass a workspace
// check; callers compare ``used`` against the workspace before carving.
struct Carve {
    uint8_t* base;
    size_t used;
    template <typename T>
    T* take(size_t count) {
        if (used > SIZE_MAX - 512 || count > (SIZE_MAX - 512 - used) / sizeof(T)) {
            used = SIZE_MAX;
            return nullptr;
        }
        T* p = base ? reinterpret_cast<T*>(base + used) : nullptr;
        used += align256(count * sizeof(T));
        return p;
    }
};

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }
static bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3) == 0; }
// a weight pointer aligned to its element (2 bytes for bf16, 4 for f32)
static bool aligned_elem(const void* p, mc_dtype dt) {
    return (reinterpret_cast<uintptr_t>(p) & (dt == MC_BF16 ? 1u : 3u)) == 0;
}

// Projection D = A W with W [K][N] row-major (the MN-major B operand);
// A and W both bf16 (f16 = 0) or both fp16 (f16 = 1); D stored in fp16.
static bool weight_problem(GemmProblem& q, const void* a, int64_t a_rows, int64_t a_inner, int64_t a_ld,
                           const void* w, int64_t K, int64_t N, void* out, int64_t out_ld, int f16) {
    memset(&q, 0, sizeof(q));
    if (!make_tmap_3d(&q.tmA, a, a_inner, a_rows, 1, a_ld, 0, kBK, kBM, f16)) return false;
    if (!make_tmap_3d(&q.tmB, w, N, K, 1, N, 0, 64, kStageKPair, f16)) return false;
    q.ab_f16 = f16;
    q.out_kind = kOutF16;
    q.M = (int)a_rows;
    q.N = (int)N;
    q.K = (int)K;
    q.batch = 1;
    q.b_mn = 1;
    q.out = out;
    q.out_ld = out_ld;
    q.out_bstride = 0;
    q.alpha = 1.f;
    q.beta = 0.f;
    q.vec_ok = (out_ld % 8 == 0) && aligned16(out);
    // fp16 output chunks leave through one TMA tensor store each
    q.bulk_st = q.vec_ok && make_tmap_3d(&q.tmC, out, N, a_rows, 1, out_ld, 0, 64, 32, 1);
    return true;
}

}  // namespace mc

using namespace mc;

#define MC_CUDA(call)                                  \
    do {                                               \
        cudaError_t e_ = (call);                       \
        if (e_ != cudaSuccess) return MC_ERR_CUDA;     \
    } while (0)

extern "C" {

const char* mc_status_string(mc_status s) {
    switch (s) {
        case MC_OK: return "ok";
        case MC_ERR_INVALID_ARG: return "invalid argument";
        case MC_ERR_UNSUPPORTED: return "unsupported shape or type";
        case MC_ERR_CUDA: return "CUDA error";
        case MC_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    }
    return "unknown status";
}

mc_status mc_read_device_status(mc_stream_t stream, unsigned* bits, int clear) {
    if (!bits) return MC_ERR_INVALID_ARG;
    MC_CUDA(cudaStreamSynchronize((cudaStream_t)stream));
    unsigned* p = device_status_ptr();
    if (!p) return MC_ERR_CUDA;
    MC_CUDA(cudaMemcpy(bits, p, sizeof(unsigned), cudaMemcpyDeviceToHost));
    if (clear) MC_CUDA(cudaMemset(p, 0, sizeof(unsigned)));
    return MC_OK;
}

mc_status mc_selftest_wait_timeout(unsigned limit_us, long long* out, mc_stream_t stream) {
    if (limit_us < 1 || limit_us > 1000000u || !out || (reinterpret_cast<uintptr_t>(out) & 7))
        return MC_ERR_INVALID_ARG;
    MC_CUDA(launch_wait_selftest((uint64_t)limit_us * 1000ull, out, (cudaStream_t)stream));
    return MC_OK;
}

unsigned long long mc_launch_count(void) { return g_launches.load(); }

mc_status mc_trace_enable(int on) {
    g_trace_on.store(on ? 1 : 0);
    return MC_OK;
}

int mc_trace_collect(mc_trace_entry* out, int cap, int keep) {
    std::vector<TraceRec> recs;
    {
        std::lock_guard<std::mutex> lk(g_trace_mu);
        if (keep) recs = g_trace;
        else recs.swap(g_trace);
    }
    std::map<std::string, std::pair<long long, double>> agg;
    std::vector<std::string> order;
    int rc = 0;
    for (auto& r : recs) {
        float ms = 0.f;
        if (cudaEventSynchronize(r.b) != cudaSuccess || cudaEventElapsedTime(&ms, r.a, r.b) != cudaSuccess) rc = -1;
        auto it = agg.find(r.name);
        if (it == agg.end()) {
            order.push_back(r.name);
            agg[r.name] = {1, (double)ms};
        } else {
            it->second.first += 1;
            it->second.second += ms;
        }
    }
    if (!keep) {
        std::lock_guard<std::mutex> lk(g_trace_mu);
        for (auto& r : recs) {
            g_event_pool.push_back(r.a);
            g_event_pool.push_back(r.b);
        }
    }
    if (rc) return -1;
    int n = 0;
    for (auto& name : order) {
        if (out && n < cap) {
            memset(out[n].name, 0, sizeof(out[n].name));
            strncpy(out[n].name, name.c_str(), sizeof(out[n].name) - 1);
            out[n].launches = agg[name].first;
            out[n].total_ms = agg[name].second;
        }
        ++n;
    }
    return n;
}

// ===========================================================================
// (1) max-logit scan
// ===========================================================================

static bool mha_tensor_path(mc_dtype dt, int D, int dh) { return dt == MC_BF16 && D % 8 == 0 && dh % 64 == 0 && dh <= 192; }

// The tensor-core scans and attention forwards max-merge S straight into the
// caller's s_max / s_bh with integer atomics (no pass after the kernel):
// every word starts at 0xFFFFFFFF, which sorts below every value, except
// that s_max keeps its maxima when the call accumulates.
static cudaError_t reset_smax(float* s_max, float* s_bh, int B, int H, int accumulate, cudaStream_t stream) {
    if (!accumulate) {
        cudaError_t e = cudaMemsetAsync(s_max, 0xFF, sizeof(float) * (size_t)H, stream);
        if (e != cudaSuccess) return e;
    }
    return s_bh ? cudaMemsetAsync(s_bh, 0xFF, sizeof(float) * (size_t)B * H, stream) : cudaSuccess;
}

static size_t mha_carve(Carve& c, int B, int T, int D, int H, int dh, mc_dtype dt, void** q, void** k,
                        unsigned** keys) {
    const size_t n = mul_sat((size_t)B * T, (size_t)H * dh);
    if (mha_tensor_path(dt, D, dh)) {
        *q = c.take<__half>(n);
        *k = c.take<__half>(n);
        *keys = nullptr;
    } else {
        *q = c.take<float>(n);
        *k = c.take<float>(n);
        *keys = c.take<unsigned>((size_t)B * H);  // the CUDA-core scan's per-(b, h) keys
    }
    return c.used;
}

size_t mc_attention_mha_workspace_size(int B, int H) {
    (void)B;
    (void)H;
    return 0;  // the forwards merge S_max straight into the outputs
}

mc_status mc_attention_mha(const void* q, const void* k, const void* v, int B, int T, int H, int dh, int causal,
                           int accumulate, void* o, float* s_max, float* s_max_bh, void* ws, size_t ws_bytes,
                           mc_stream_t stream_) {
    cudaStream_t stream = (cudaStream_t)stream_;
    if (!q || !k || !v || !o || !s_max) return MC_ERR_INVALID_ARG;
    if (!aligned4(s_max) || !aligned4(s_max_bh)) return MC_ERR_INVALID_ARG;  // merged into with 32-bit atomics
    if (B <= 0 || T <= 0 || H <= 0 || dh <= 0) return MC_ERR_INVALID_ARG;
    if (dh != 64 && dh != 128) return MC_ERR_UNSUPPORTED;
    if ((int64_t)B * T > INT32_MAX || (int64_t)H * dh > INT32_MAX) return MC_ERR_UNSUPPORTED;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return MC_ERR_INVALID_ARG;
    if (o == q || o == k || o == v) return MC_ERR_INVALID_ARG;
    (void)ws;  // no workspace: S_max is merged straight into s_max / s_max_bh
    (void)ws_bytes;
    MC_CUDA(reset_smax(s_max, s_max_bh, B, H, accumulate, stream));
    AttnArgs a;
    memset(&a, 0, sizeof(a));
    a.q = q;
    a.k = k;
    a.v = v;
    a.o = o;
    a.B = B;
    a.T = T;
    a.H = H;
    a.dh = dh;
    a.causal = causal ? 1 : 0;
    a.s_max = s_max;
    a.s_bh = s_max_bh;
    MC_CUDA(launch_attn(a, stream));
    return MC_OK;
}

mc_status mc_attention_mla(const void* q, const void* k_c, const void* k_r, int kr_ld, int kr_col, const void* v,
                           int B, int T, int H, int nope, int rope, int dv, int causal, int accumulate, void* o,
                           float* s_max, float* s_max_bh, void* ws, size_t ws_bytes, mc_stream_t stream_) {
    cudaStream_t stream = (cudaStream_t)stream_;
    if (!q || !k_c || !k_r || !v || !o || !s_max) return MC_ERR_INVALID_ARG;
    if (!aligned4(s_max) || !aligned4(s_max_bh)) return MC_ERR_INVALID_ARG;  // merged into with 32-bit atomics
    if (B <= 0 || T <= 0 || H <= 0 || nope <= 0 || rope <= 0 || dv <= 0) return MC_ERR_INVALID_ARG;
    if (nope != 128 || rope != 64 || dv != 128) return MC_ERR_UNSUPPORTED;
    if ((int64_t)B * T > INT32_MAX || (int64_t)H * 192 > INT32_MAX) return MC_ERR_UNSUPPORTED;
    if (kr_col < 0 || kr_ld < kr_col + rope || kr_ld % 8 || kr_col % 8) return MC_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_c) || !aligned16(k_r) || !aligned16(v) || !aligned16(o)) return MC_ERR_INVALID_ARG;
    if (o == q || o == k_c || o == k_r || o == v) return MC_ERR_INVALID_ARG;
    (void)ws;  // no workspace: S_max is merged straight into s_max / s_max_bh
    (void)ws_bytes;
    MC_CUDA(reset_smax(s_max, s_max_bh, B, H, accumulate, stream));
    AttnArgs a;
    memset(&a, 0, sizeof(a));
    a.q = q;
    a.k = k_c;
    a.v = v;
    a.kr = k_r;
    a.kr_ld = kr_ld;
    a.kr_col = kr_col;
    a.mla = 1;
    a.o = o;
    a.B = B;
    a.T = T;
    a.H = H;
    a.dh = nope + rope;
    a.causal = causal ? 1 : 0;
    a.s_max = s_max;
    a.s_bh = s_max_bh;
    MC_CUDA(launch_attn(a, stream));
    return MC_OK;
}

size_t mc_max_logits_mha_workspace_size(int B, int T, int D, int H, int dh, mc_dtype dtype) {
    if (B <= 0 || T <= 0 || D <= 0 || H <= 0 || dh <= 0) return 0;
    Carve c{nullptr, 0};
    void *q, *k;
    unsigned* keys;
    return mha_carve(c, B, T, D, H, dh, dtype, &q, &k, &keys);
}

mc_status mc_max_logits_mha(const void* x, const void* wq, const void* wk, mc_dtype dtype, int B, int T, int D,
                            int H, int dh, int causal, int accumulate, float* s_max, float* s_max_bh, void* ws,
                            size_t ws_bytes, mc_stream_t stream_) {
    cudaStream_t stream = (cudaStream_t)stream_;
    if (!x || !wq || !wk || !s_max) return MC_ERR_INVALID_ARG;
    if (!aligned4(s_max) || !aligned4(s_max_bh)) return MC_ERR_INVALID_ARG;  // merged into with 32-bit atomics
    if (B <= 0 || T <= 0 || D <= 0 || H <= 0 || dh <= 0) return MC_ERR_INVALID_ARG;
    if (dtype != MC_F32 && dtype != MC_BF16) return MC_ERR_INVALID_ARG;
    if (!aligned_elem(x, dtype) || !aligned_elem(wq, dtype) || !aligned_elem(wk, dtype)) return MC_ERR_INVALID_ARG;
    if ((int64_t)B * T > INT32_MAX || (int64_t)H * dh > INT32_MAX) return MC_ERR_UNSUPPORTED;
    size_t need = mc_max_logits_mha_workspace_size(B, T, D, H, dh, dtype);
    if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255) || ws_bytes < need) return MC_ERR_WORKSPACE;
    Carve c{(uint8_t*)ws, 0};
    void *q, *k;
    unsigned* keys;
    mha_carve(c, B, T, D, H, dh, dtype, &q, &k, &keys);
    const int64_t BT = (int64_t)B * T, N = (int64_t)H * dh;
    if (mha_tensor_path(dtype, D, dh)) {
        MC_CUDA(reset_smax(s_max, s_max_bh, B, H, accumulate, stream));
        if (!aligned16(x) || !aligned16(wq) || !aligned16(wk)) return MC_ERR_INVALID_ARG;
        GemmParams P;
        memset(&P, 0, sizeof(P));
        P.nprob = 2;
        if (!weight_problem(P.p[0], x, BT, D, D, wq, D, N, q, N, 0)) return MC_ERR_INVALID_ARG;
        if (!weight_problem(P.p[1], x, BT, D, D, wk, D, N, k, N, 0)) return MC_ERR_INVALID_ARG;
        P.tile_m = kPairTileM;
        P.a_shared = 1;
        finalize_gemm_params(P);
        MC_CUDA(launch_gemm(P, stream, "gemm:proj"));
        ScanArgs a;
        memset(&a, 0, sizeof(a));
        a.q = q;
        a.q_ld = N;
        a.k = k;
        a.k_ld = N;
        a.B = B;
        a.T = T;
        a.H = H;
        a.causal = causal ? 1 : 0;
        a.q_head_stride = dh;
        a.k_head_stride = dh;
        a.nkb_main = dh / 64;
        a.nkb_rope = 0;
        a.d = (float)dh;
        a.s_max = s_max;
        a.s_bh = s_max_bh;
        MC_CUDA(launch_scan(a, stream));  // merges S into s_max / s_max_bh
    } else {
        MC_CUDA(cudaMemsetAsync(keys, 0, sizeof(unsigned) * (size_t)B * H, stream));
        MC_CUDA(launch_proj_simt(x, wq, dtype, (float*)q, (int)BT, D, (int)N, stream));
        MC_CUDA(launch_proj_simt(x, wk, dtype, (float*)k, (int)BT, D, (int)N, stream));
        MC_CUDA(launch_scan_simt((const float*)q, (const float*)k, B, T, H, dh, causal ? 1 : 0, keys, stream));
        MC_CUDA(launch_finalize_smax(keys, B, H, (float)dh, accumulate, s_max, s_max_bh, stream));
    }
    return MC_OK;
}

// ---------------------------------------------------------------------------
// Allocation-free scan: the scratch is a static device array of the library
// (one per device that loads it), so callers that may not allocate -- plugins
// in frameworks that own all device memory, code running under stream
// capture -- can still run the scan.  Its device address is looked up once
// per device; all calls share the array, so overlapping calls race.
// ---------------------------------------------------------------------------
static __device__ __align__(256) unsigned char g_noalloc_scratch[MC_NOALLOC_SCRATCH_BYTES];
static void* g_noalloc_ptr[64];

static void* noalloc_scratch() {
    int dev = current_device();
    if (dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_noalloc_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
        g_noalloc_ptr[dev] = p;
    }
    return g_noalloc_ptr[dev];
}

mc_status mc_max_logits_mha_noalloc(const void* x, const void* wq, const void* wk, mc_dtype dtype, int B, int T,
                                    int D, int H, int dh, int causal, int accumulate, float* s_max,
                                    float* s_max_bh, mc_stream_t stream) {
    if (B <= 0 || T <= 0 || D <= 0 || H <= 0 || dh <= 0) return MC_ERR_INVALID_ARG;
    if ((int64_t)B * T > INT32_MAX || (int64_t)H * dh > INT32_MAX) return MC_ERR_UNSUPPORTED;
    if (mc_max_logits_mha_workspace_size(B, T, D, H, dh, dtype) > MC_NOALLOC_SCRATCH_BYTES) return MC_ERR_WORKSPACE;
    void* scratch = noalloc_scratch();
    if (!scratch) return MC_ERR_CUDA;
    return mc_max_logits_mha(x, wq, wk, dtype, B, T, D, H, dh, causal, accumulate, s_max, s_max_bh, scratch,
                             MC_NOALLOC_SCRATCH_BYTES, stream);
}

static mc_status mla_check(const mc_mla_layer* L, bool scan) {
    if (!L) return MC_ERR_INVALID_ARG;
    if (L->D <= 0 || L->q_lora <= 0 || L->kv_lora <= 0 || L->H <= 0 || L->nope < 0 || L->rope < 0)
        return MC_ERR_INVALID_ARG;
    if (!L->w_qb || !L->w_kb) return MC_ERR_INVALID_ARG;
    if (L->wtype != MC_BF16 && L->wtype != MC_F32) return MC_ERR_INVALID_ARG;
    if (scan) {
        if (!L->w_qa || !L->w_kva) return MC_ERR_INVALID_ARG;
        if (L->wtype != MC_BF16 || L->rope != 64 || L->nope % 64 || L->nope <= 0 || L->nope + L->rope > 192 ||
            L->D % 64 || L->q_lora % 64 || L->kv_lora % 64)
            return MC_ERR_UNSUPPORTED;
    }
    return MC_OK;
}

struct MlaWs {
    float2* rope;
    __half *cq, *ckv, *q, *kc, *wqb, *wkb;  // fp16 intermediates and fp16 copies of W_qb, W_kb
};

static size_t mla_carve(Carve& c, const mc_mla_layer* L, int B, int T, MlaWs& w) {
    size_t BT = (size_t)B * T;
    w.rope = c.take<float2>((size_t)T * 32);
    const size_t H = (size_t)L->H, qk = (size_t)L->nope + L->rope;
    w.cq = c.take<__half>(mul_sat(BT, L->q_lora));
    w.ckv = c.take<__half>(mul_sat(BT, (size_t)L->kv_lora + L->rope));
    w.q = c.take<__half>(mul_sat(BT, H, qk));
    w.kc = c.take<__half>(mul_sat(BT, H, L->nope));
    w.wqb = c.take<__half>(mul_sat(L->q_lora, H, qk));
    w.wkb = c.take<__half>(mul_sat(L->kv_lora, H, L->nope));
    return c.used;
}

size_t mc_max_logits_mla_workspace_size(const mc_mla_layer* L, int B, int T) {
    if (!L || B <= 0 || T <= 0 || L->H <= 0) return 0;
    Carve c{nullptr, 0};
    MlaWs w;
    return mla_carve(c, L, B, T, w);
}

mc_status mc_max_logits_mla(const mc_mla_layer* L, const void* x, int B, int T, int causal, int accumulate,
                            float* s_max, float* s_max_bh, void* ws, size_t ws_bytes, mc_stream_t stream_) {
    cudaStream_t stream = (cudaStream_t)stream_;
    mc_status st = mla_check(L, true);
    if (st != MC_OK) return st;
    if (!x || !s_max || B <= 0 || T <= 0) return MC_ERR_INVALID_ARG;
    if (!aligned4(s_max) || !aligned4(s_max_bh)) return MC_ERR_INVALID_ARG;  // merged into with 32-bit atomics
    if ((int64_t)B * T > INT32_MAX) return MC_ERR_UNSUPPORTED;
    if (!aligned16(x) || !aligned16(L->w_qa) || !aligned16(L->w_qb) || !aligned16(L->w_kva) || !aligned16(L->w_kb))
        return MC_ERR_INVALID_ARG;
    size_t need = mc_max_logits_mla_workspace_size(L, B, T);
    if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255) || ws_bytes < need) return MC_ERR_WORKSPACE;
    Carve c{(uint8_t*)ws, 0};
    MlaWs w;
    mla_carve(c, L, B, T, w);
    const int64_t BT = (int64_t)B * T;
    const int qk = L->nope + L->rope, kvw = L->kv_lora + L->rope;
    MC_CUDA(reset_smax(s_max, s_max_bh, B, L->H, accumulate, stream));
    MC_CUDA(launch_rope_table(w.rope, T, L->rope_base, stream));
    // phase 1: c_Q = x W_qa ; [c_KV | k^R] = x W_kva (RoPE on the k^R columns)
    GemmParams P;
    memset(&P, 0, sizeof(P));
    P.nprob = 2;
    if (!weight_problem(P.p[0], x, BT, L->D, L->D, L->w_qa, L->D, L->q_lora, w.cq, L->q_lora, 0))
        return MC_ERR_INVALID_ARG;
    if (!weight_problem(P.p[1], x, BT, L->D, L->D, L->w_kva, L->D, kvw, w.ckv, kvw, 0)) return MC_ERR_INVALID_ARG;
    P.p[1].rope_tab = w.rope;
    P.p[1].rope_T = T;
    P.p[1].rope_period = kvw;
    P.p[1].rope_start = L->kv_lora;
    P.tile_m = kPairTileM;
    P.a_shared = 1;
    finalize_gemm_params(P);
    MC_CUDA(launch_gemm(P, stream, "gemm:proj"));
    // phase 2: [q^C | q^R] = c_Q W_qb (RoPE on q^R) ; k^C = c_KV W_kb, on
    // fp16 operands (W_qb, W_kb converted; exact in fp16's normal range)
    const int64_t Nq = (int64_t)L->H * qk, Nk = (int64_t)L->H * L->nope;
    MC_CUDA(launch_bf16_to_f16(L->w_qb, w.wqb, (long long)L->q_lora * Nq, stream));
    MC_CUDA(launch_bf16_to_f16(L->w_kb, w.wkb, (long long)L->kv_lora * Nk, stream));
    memset(&P, 0, sizeof(P));
    P.nprob = 2;
    if (!weight_problem(P.p[0], w.cq, BT, L->q_lora, L->q_lora, w.wqb, L->q_lora, Nq, w.q, Nq, 1))
        return MC_ERR_INVALID_ARG;
    P.p[0].rope_tab = w.rope;
    P.p[0].rope_T = T;
    P.p[0].rope_period = qk;
    P.p[0].rope_start = L->nope;
    if (!weight_problem(P.p[1], w.ckv, BT, L->kv_lora, kvw, w.wkb, L->kv_lora, Nk, w.kc, Nk, 1))
        return MC_ERR_INVALID_ARG;
    P.tile_m = kPairTileM;
    finalize_gemm_params(P);
    MC_CUDA(launch_gemm(P, stream, "gemm:proj"));
    // scan: per head 3 K blocks (q^C.k^C x2, q^R.k^R x1)
    ScanArgs a;
    memset(&a, 0, sizeof(a));
    a.q = w.q;
    a.q_ld = Nq;
    a.k = w.kc;
    a.k_ld = Nk;
    a.kr = w.ckv;
    a.kr_ld = kvw;
    a.B = B;
    a.T = T;
    a.H = L->H;
    a.causal = causal ? 1 : 0;
    a.q_head_stride = qk;
    a.k_head_stride = L->nope;
    a.nkb_main = L->nope / 64;
    a.nkb_rope = 1;
    a.kr_col = L->kv_lora;
    a.d = (float)qk;
    a.s_max = s_max;
    a.s_bh = s_max_bh;
    MC_CUDA(launch_scan(a, stream));  // merges S into s_max / s_max_bh
    return MC_OK;
}

// ===========================================================================
// (2) QK-Clip
// ===========================================================================

mc_status mc_qk_clip_mha(void* wq, void* wk, mc_dtype dtype, int D, int H, int dh, const float* s_max, float tau,
                         float* gamma, mc_stream_t stream) {
    if (!wq || !wk || !s_max || D <= 0 || H <= 0 || dh <= 0) return MC_ERR_INVALID_ARG;
    if (dtype != MC_F32 && dtype != MC_BF16) return MC_ERR_INVALID_ARG;
    if (!aligned_elem(wq, dtype) || !aligned_elem(wk, dtype) || !aligned4(s_max) || !aligned4(gamma))
        return MC_ERR_INVALID_ARG;
    ClipArgs a;
    memset(&a, 0, sizeof(a));
    a.nseg = 2;
    a.H = H;
    a.bf16 = dtype == MC_BF16;
    a.s_max = s_max;
    a.tau = tau;
    a.gamma_out = gamma;
    for (int s = 0; s < 2; ++s) {
        a.seg[s].w = s ? wk : wq;
        a.seg[s].ld = (long long)H * dh;
        a.seg[s].rows = D;
        a.seg[s].col0 = 0;
        a.seg[s].head_stride = dh;
        a.seg[s].width = dh;
        a.seg[s].use_gamma = 0;
    }
    MC_CUDA(launch_clip(a, (cudaStream_t)stream));
    return MC_OK;
}

mc_status mc_qk_clip_mla(const mc_mla_layer* L, const float* s_max, float tau, float* gamma, mc_stream_t stream) {
    mc_status st = mla_check(L, false);
    if (st != MC_OK) return st;
    if (!s_max) return MC_ERR_INVALID_ARG;
    if (!aligned_elem(L->w_qb, (mc_dtype)L->wtype) || !aligned_elem(L->w_kb, (mc_dtype)L->wtype) || !aligned4(s_max) ||
        !aligned4(gamma))
        return MC_ERR_INVALID_ARG;
    const int qk = L->nope + L->rope;
    ClipArgs a;
    memset(&a, 0, sizeof(a));
    a.H = L->H;
    a.bf16 = L->wtype == MC_BF16;
    a.s_max = s_max;
    a.tau = tau;
    a.gamma_out = gamma;
    int n = 0;
    if (L->nope > 0) {  // q^C x sqrt(gamma)
        a.seg[n++] = ClipSeg{L->w_qb, (long long)L->H * qk, L->q_lora, 0, qk, L->nope, 0};
    }
    if (L->rope > 0) {  // q^R x gamma
        a.seg[n++] = ClipSeg{L->w_qb, (long long)L->H * qk, L->q_lora, L->nope, qk, L->rope, 1};
    }
    if (L->nope > 0) {  // k^C x sqrt(gamma)
        a.seg[n++] = ClipSeg{L->w_kb, (long long)L->H * L->nope, L->kv_lora, 0, L->nope, L->nope, 0};
    }
    a.nseg = n;
    if (n == 0) return MC_OK;
    MC_CUDA(launch_clip(a, (cudaStream_t)stream));
    return MC_OK;
}

mc_status mc_qk_clip_global(void* wq, void* wk, mc_dtype dtype, int rows, int cols, const float* s_max, int H,
                            float tau, float alpha, float* gamma_out, mc_stream_t stream) {
    if (!wq || !wk || !s_max || rows <= 0 || cols <= 0 || H <= 0) return MC_ERR_INVALID_ARG;
    if (dtype != MC_F32 && dtype != MC_BF16) return MC_ERR_INVALID_ARG;
    if (!aligned_elem(wq, dtype) || !aligned_elem(wk, dtype) || !aligned4(s_max) || !aligned4(gamma_out))
        return MC_ERR_INVALID_ARG;
    MC_CUDA(launch_clip_global(wq, wk, dtype == MC_BF16, (long long)rows * cols, s_max, H, tau, alpha, gamma_out,
                               (cudaStream_t)stream));
    return MC_OK;
}

// ===========================================================================
// (3) Muon
// ===========================================================================

namespace {

struct NsGroup {
    int m, n, m_pad, n_pad;
    std::vector<int> idx;  // input indices
    int zbase;             // position of idx[0] in the group-ordered list
    __nv_bfloat16* X[2];
    __nv_bfloat16* A;
    __nv_bfloat16* Bm;
};

struct NsPlan {
    std::vector<NsGroup> groups;
    std::vector<int> order;      // group-ordered input indices
    std::vector<double*> part;   // per ordered position
    std::vector<int> nparts;
    float* s;
    float* s2;
    unsigned* bar;  // grid-barrier counter of the multi-phase launches
    MatInfo* info;  // per-matrix facts, written by the momentum pass
    size_t bytes;
};

int round_up(int v, int m) { return (v + m - 1) / m * m; }

bool plan_ns(const int* rows, const int* cols, int count, uint8_t* base, NsPlan& P) {
    P.groups.clear();
    P.order.clear();
    for (int i = 0; i < count; ++i) {
        int m = std::min(rows[i], cols[i]), n = std::max(rows[i], cols[i]);
        int mp = round_up(m, 256), np = round_up(n, 64);
        int g = -1;
        for (size_t j = 0; j < P.groups.size(); ++j)
            if (P.groups[j].m_pad == mp && P.groups[j].n_pad == np) g = (int)j;
        if (g < 0) {
            NsGroup ng;
            ng.m = m;
            ng.n = n;
            ng.m_pad = mp;
            ng.n_pad = np;
            P.groups.push_back(ng);
            g = (int)P.groups.size() - 1;
        }
        P.groups[g].idx.push_back(i);
    }
    Carve c{base, 0};
    for (auto& g : P.groups) {
        g.zbase = (int)P.order.size();
        for (int i : g.idx) P.order.push_back(i);
        size_t cnt = g.idx.size();
        g.X[0] = c.take<__nv_bfloat16>(mul_sat(cnt, g.m_pad, g.n_pad));
        g.X[1] = c.take<__nv_bfloat16>(mul_sat(cnt, g.m_pad, g.n_pad));
        g.A = c.take<__nv_bfloat16>(mul_sat(cnt, g.m_pad, g.m_pad));
        g.Bm = c.take<__nv_bfloat16>(mul_sat(cnt, g.m_pad, g.m_pad));
    }
    P.part.assign(count, nullptr);
    P.nparts.assign(count, 0);
    for (auto& g : P.groups)
        for (size_t k = 0; k < g.idx.size(); ++k) {
            int np = (g.m_pad / 64) * (g.n_pad / 64);
            P.part[g.zbase + k] = c.take<double>(np);
            P.nparts[g.zbase + k] = np;
        }
    P.s = c.take<float>(count);
    P.s2 = c.take<float>(count);
    P.bar = c.take<unsigned>(1);
    P.info = c.take<MatInfo>(count);
    P.bytes = c.used;
    return true;
}

bool valid_mats(const int* rows, const int* cols, int count) {
    if (!rows || !cols || count <= 0) return false;
    for (int i = 0; i < count; ++i) {
        if (rows[i] <= 0 || cols[i] <= 0) return false;
        if (rows[i] > (1 << 30) || cols[i] > (1 << 30)) return false;  // padded sizes stay in int
        if ((int64_t)rows[i] * cols[i] > ((int64_t)1 << 31)) return false;
    }
    return true;
}

// mode 0/1: momentum (+ cast) or cast; mode 2/3: update or write O
mc_status run_mat_pass(const NsPlan& P, int mode, float* const* w, const float* const* g, float* const* m,
                       const float* const* in, const int* rows, const int* cols, int xbuf, float mu, float lr,
                       float wd, float rms_coef, int nesterov, bool zero_steps, cudaStream_t stream) {
    const int count = (int)P.order.size();
    // position -> group
    std::vector<const NsGroup*> grp(count);
    std::vector<int> within(count);
    for (auto& gr : P.groups)
        for (size_t k = 0; k < gr.idx.size(); ++k) {
            grp[gr.zbase + k] = &gr;
            within[gr.zbase + k] = (int)k;
        }
    for (int c0 = 0; c0 < count; c0 += kMaxBatchMats) {
        MatBatch B;
        memset(&B, 0, sizeof(B));
        B.mode = mode;
        B.mu = mu;
        B.lr = lr;
        B.wd = wd;
        B.nesterov = nesterov;
        B.x_f16 = mode >= 2 && !zero_steps ? 1 : 0;
        B.info = mode <= 1 ? P.info : nullptr;
        B.info_base = c0;
        int tiles = 0;
        for (int p = c0; p < std::min(count, c0 + kMaxBatchMats); ++p) {
            const int i = P.order[p];
            const NsGroup& gr = *grp[p];
            MatDesc& d = B.d[B.count++];
            d.rows = rows[i];
            d.cols = cols[i];
            d.tr = rows[i] > cols[i];
            d.m_pad = gr.m_pad;
            d.n_pad = gr.n_pad;
            d.x = gr.X[xbuf] + (size_t)within[p] * gr.m_pad * gr.n_pad;
            d.partial = P.part[p];
            d.tiles_x = gr.n_pad / 64;
            d.tile_begin = tiles;
            tiles += (gr.m_pad / 64) * (gr.n_pad / 64);
            d.w = w[i];
            d.rms = rms_coef * sqrtf((float)std::max(rows[i], cols[i]));
            // float4 accesses need whole 16-byte groups of columns on every row
            d.vec = cols[i] % 4 == 0 &&
                    (mode == 0 ? aligned16(m[i]) && aligned16(g[i])
                               : mode == 1 ? aligned16(in[i]) : aligned16(w[i]));
            d.flat = d.vec && !d.tr && gr.m_pad == rows[i] && gr.n_pad == cols[i];
            if (mode == 0) {
                d.m = m[i];
                d.g = g[i];
            } else if (mode == 1) {
                d.m = const_cast<float*>(in[i]);
            } else {
                d.oscale = zero_steps ? P.s + p : nullptr;
            }
        }
        B.total_tiles = tiles;
        MC_CUDA(launch_mat_pass(B, stream));
    }
    return MC_OK;
}

mc_status run_norm(const NsPlan& P, float eps, cudaStream_t stream) {
    const int count = (int)P.order.size();
    for (int c0 = 0; c0 < count; c0 += kMaxBatchMats) {
        NormArgs a;
        memset(&a, 0, sizeof(a));
        a.eps = eps;
        a.s = P.s + c0;
        a.s2 = P.s2 + c0;
        for (int p = c0; p < std::min(count, c0 + kMaxBatchMats); ++p) {
            a.partial[a.count] = P.part[p];
            a.nparts[a.count] = P.nparts[p];
            ++a.count;
        }
        MC_CUDA(launch_norm_finalize(a, stream));
    }
    return MC_OK;
}

// One Newton-Schulz GEMM of iteration `it` for a shape group:
// kind 0: Gram A = sc2 X X^T ; 1: poly B = c A A + b A ; 2: apply X' = sc (B X + a X).
// sym: Gram and poly compute the tiles on and above the diagonal and mirror
// them (exactly symmetric A, B); otherwise every tile is computed, which
// costs no time when the full tiling still fits the same number of waves.
bool ns_problem(GemmProblem& q, const NsPlan& P, const NsGroup& gr, int kind, int it, float a, float b,
                float c, int bn, int sym, int tile_m) {
    const uint32_t brows = tile_m == kBM ? bn : bn / 2;  // K-major B rows loaded per CTA
    memset(&q, 0, sizeof(q));
    const int xin = it & 1, xout = (it + 1) & 1;
    const uint64_t cnt = gr.idx.size(), mp = gr.m_pad, np = gr.n_pad;
    q.batch = (int)cnt;
    q.vec_ok = 1;
    // Number formats.  The momentum pass writes X unscaled in bf16 (any
    // magnitude fits).  Every later X, A and B is bounded (normalised X,
    // |entries| below about 12), and those are held in fp16: its 11
    // significant bits keep the iteration within a few 1e-3 of the fp64
    // result where bf16's 8 reached 2e-2 on thin matrices.  Both operands of
    // one MMA share a type, so the first iteration converts on its outputs:
    //   Gram 0  bf16 X  -> fp16 A (scaled by s^2)
    //   poly 0  fp16 A  -> bf16 B (B meets the bf16 X in the apply)
    //   apply 0 bf16 B, X -> fp16 X (scaled by s)
    // and every later GEMM reads and writes fp16.
    // The apply X' = aX + BX reads X a second time, as the epilogue's aux.
    // From the second iteration on, the poly adds a to its diagonal instead
    // (B' = aI + B, the same product: X' = B'X), so the apply is a plain
    // product whose epilogue reads nothing beside its accumulator.  Its
    // entries round in fp16 once, at most 2^-10 on a diagonal below 4, less
    // than X's own fp16 rounding.  The first apply keeps aX0 in fp32 from the
    // unscaled bf16 X0, whose B is bf16 (a + B_ii would lose 2^-7 there).
    const int in_f16 = it == 0 ? (kind == 1) : 1;
    const int out_f16 = it == 0 ? (kind != 1) : 1;
    q.ab_f16 = in_f16;  // the aux operand (A in poly, X in apply) has the same type
    q.out_kind = out_f16 ? kOutF16 : kOutBF16;
    // workspace buffers: 256-byte aligned, rows of m_pad / n_pad (multiples of 64) elements
    q.bulk_st = kind == 2 || !sym;
    // symmetric Gram and poly outputs: their chunks above the diagonal go out
    // by TMA stores too, the rows and (transposed by a pair of warps) the mirror
    q.sym_tma = sym && kind != 2;
    if (q.bulk_st || q.sym_tma) {
        const void* out = kind == 0 ? (const void*)gr.A : kind == 1 ? (const void*)gr.Bm : (const void*)gr.X[xout];
        const uint64_t on = kind == 2 ? np : mp;
        if (!make_tmap_3d(&q.tmC, out, on, mp, cnt, on, mp * on, 64, 32, out_f16)) return false;
    }
    if (kind == 0) {
        if (!make_tmap_3d(&q.tmA, gr.X[xin], np, mp, cnt, np, mp * np, kBK, kBM, in_f16)) return false;
        if (!make_tmap_3d(&q.tmB, gr.X[xin], np, mp, cnt, np, mp * np, kBK, brows, in_f16)) return false;
        q.M = q.N = (int)mp;
        q.K = (int)np;
        q.sym = sym;
        q.out = gr.A;
        q.out_ld = mp;
        q.out_bstride = mp * mp;
        q.alpha = 1.f;
        q.scale = it == 0 ? P.s2 + gr.zbase : nullptr;
    } else if (kind == 1) {
        if (!make_tmap_3d(&q.tmA, gr.A, mp, mp, cnt, mp, mp * mp, kBK, kBM, in_f16)) return false;
        if (!make_tmap_3d(&q.tmB, gr.A, mp, mp, cnt, mp, mp * mp, kBK, brows, in_f16)) return false;
        q.M = q.N = q.K = (int)mp;
        q.sym = sym;
        q.out = gr.Bm;
        q.out_ld = mp;
        q.out_bstride = mp * mp;
        q.aux = gr.A;
        q.aux_ld = mp;
        q.aux_bstride = mp * mp;
        q.alpha = c;
        q.beta = b;
        if (it > 0) q.diag = a;  // B' = aI + bA + cA^2
    } else {
        if (!make_tmap_3d(&q.tmA, gr.Bm, mp, mp, cnt, mp, mp * mp, kBK, kBM, in_f16)) return false;
        if (!make_tmap_3d(&q.tmB, gr.X[xin], np, mp, cnt, np, mp * np, 64, stage_k_for(tile_m), in_f16))
            return false;
        q.b_mn = 1;
        q.M = (int)mp;
        q.N = (int)np;
        q.K = (int)mp;
        q.out = gr.X[xout];
        q.out_ld = np;
        q.out_bstride = mp * np;
        q.alpha = 1.f;
        if (it == 0) {  // X1 = s (a X0 + B X0)
            q.aux = gr.X[xin];
            q.aux_ld = np;
            q.aux_bstride = mp * np;
            q.beta = a;
            q.scale = P.s + gr.zbase;
        }  // later: X' = B' X
    }
    return true;
}

// All Newton-Schulz iterations: for every (up to 4) shape groups, up to 5
// iterations (15 phases: Gram, poly, apply) per cooperative launch, with a
// grid barrier between phases.
mc_status run_ns_iterations(const NsPlan& P, int steps, float a, float b, float c, float eps,
                            cudaStream_t stream) {
    const int ngroups = (int)P.groups.size();
    for (int g0 = 0; g0 < ngroups; g0 += 4) {
        const int g1 = std::min(ngroups, g0 + 4);
        const int per_launch = std::min(kMaxPhases / 3, kMaxProblemsMulti / (3 * (g1 - g0)));
        // Large batches: 256 x 256 tiles computed by CTA pairs (m_pad is a
        // multiple of 256).  Batches whose apply phase has fewer such tiles
        // than SM pairs: 128 x 128 tiles on single CTAs, where the pairs'
        // cross-SM hand-offs cost more than the halved B loads save.
        long long apply_tiles = 0;
        for (int g = g0; g < g1; ++g) {
            const NsGroup& gr = P.groups[g];
            apply_tiles += (long long)gr.idx.size() * (gr.m_pad / kPairTileM) * ((gr.n_pad + kBN - 1) / kBN);
        }
        const bool small = apply_tiles < num_sms() / 2;
        const int bn = small ? 128 : kBN;
        const int tile_m = small ? kBM : kPairTileM;
        const long long nsm = small ? num_sms() : num_sms() / 2;  // scheduling units
        // full Gram / poly tilings when they take no more waves than the symmetric ones
        long long sym_tiles = 0, full_tiles = 0;
        for (int g = g0; g < g1; ++g) {
            const NsGroup& gr = P.groups[g];
            const long long tm = gr.m_pad / tile_m, tn = (gr.m_pad + bn - 1) / bn;
            long long t = 0;
            for (long long i = 0; i < tm; ++i) t += tn - (tile_m * i) / bn;
            sym_tiles += (long long)gr.idx.size() * t;
            full_tiles += (long long)gr.idx.size() * tm * tn;
        }
        const int sym = (full_tiles + nsm - 1) / nsm > (sym_tiles + nsm - 1) / nsm ? 1 : 0;
        for (int it0 = 0; it0 < steps; it0 += per_launch) {
            const int nit = std::min(per_launch, steps - it0);
            static GemmParamsMulti G;  // ~27 KB: not on the stack; filled and launched under g_launch_mu
            std::lock_guard<std::mutex> lk(g_launch_mu);
            memset(&G, 0, sizeof(G));
            G.bn = bn;
            G.tile_m = tile_m;
            for (int it = it0; it < it0 + nit; ++it)
                for (int kind = 0; kind < 3; ++kind) {
                    G.phase_prob[G.nphase++] = G.nprob;
                    for (int g = g0; g < g1; ++g)
                        if (!ns_problem(G.p[G.nprob++], P, P.groups[g], kind, it, a, b, c, bn, sym, tile_m))
                            return MC_ERR_CUDA;
                }
            G.phase_prob[G.nphase] = G.nprob;
            G.grid_bar = P.bar;
            G.mats = P.info;
            G.s = P.s;
            G.s2 = P.s2;
            G.eps = eps;
            if (it0 == 0) {  // first launch of this chunk: the norm pre-phase
                G.norm_begin = P.groups[g0].zbase;
                G.norm_end = P.groups[g1 - 1].zbase + (int)P.groups[g1 - 1].idx.size();
            }
            finalize_gemm_params(G);
            MC_CUDA(cudaMemsetAsync(P.bar, 0, sizeof(unsigned), stream));
            MC_CUDA(launch_gemm_multi(G, stream, "gemm:ns"));
        }
    }
    return MC_OK;
}

mc_status muon_impl(bool step, float* const* w, const float* const* g, float* const* m, const float* const* in,
                    float* const* out, const int* rows, const int* cols, int count, float lr, float mu, float wd,
                    float rms_coef, int steps, float a, float b, float c, float eps, int nesterov, void* ws,
                    size_t ws_bytes, cudaStream_t stream) {
    if (!valid_mats(rows, cols, count) || steps < 0) return MC_ERR_INVALID_ARG;
    for (int i = 0; i < count; ++i) {
        if (step) {
            if (!w || !g || !m || !w[i] || !g[i] || !m[i]) return MC_ERR_INVALID_ARG;
            if (!aligned4(w[i]) || !aligned4(g[i]) || !aligned4(m[i])) return MC_ERR_INVALID_ARG;
        } else {
            if (!in || !out || !in[i] || !out[i]) return MC_ERR_INVALID_ARG;
            if (!aligned4(in[i]) || !aligned4(out[i]) || in[i] == out[i]) return MC_ERR_INVALID_ARG;
        }
    }
    NsPlan P;
    plan_ns(rows, cols, count, nullptr, P);
    if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255) || ws_bytes < P.bytes) return MC_ERR_WORKSPACE;
    plan_ns(rows, cols, count, (uint8_t*)ws, P);
    mc_status st = run_mat_pass(P, step ? 0 : 1, step ? w : out, g, m, in, rows, cols, 0, mu, lr, wd, rms_coef,
                                nesterov, false, stream);
    if (st != MC_OK) return st;
    // the norm runs as the pre-phase of the first Newton-Schulz launch; with
    // zero steps it is a launch of its own and the update applies the scale
    if (steps > 0)
        st = run_ns_iterations(P, steps, a, b, c, eps, stream);
    else
        st = run_norm(P, eps, stream);
    if (st != MC_OK) return st;
    return run_mat_pass(P, step ? 2 : 3, step ? w : out, g, m, in, rows, cols, steps & 1, mu, lr, wd, rms_coef,
                        nesterov, steps == 0, stream);
}

}  // namespace

size_t mc_newton_schulz_workspace_size(const int* rows, const int* cols, int count) {
    if (!valid_mats(rows, cols, count)) return 0;
    NsPlan P;
    plan_ns(rows, cols, count, nullptr, P);
    return P.bytes;
}

size_t mc_muon_workspace_size(const int* rows, const int* cols, int count) {
    return mc_newton_schulz_workspace_size(rows, cols, count);
}

mc_status mc_newton_schulz(const float* const* in, float* const* out, const int* rows, const int* cols, int count,
                           int steps, float a, float b, float c, float eps, void* ws, size_t ws_bytes,
                           mc_stream_t stream) {
    return muon_impl(false, nullptr, nullptr, nullptr, in, out, rows, cols, count, 0.f, 0.f, 0.f, 0.f, steps, a, b,
                     c, eps, 0, ws, ws_bytes, (cudaStream_t)stream);
}

mc_status mc_muon_step(float* const* w, const float* const* g, float* const* m, const int* rows, const int* cols,
                       int count, float lr, float mu, float wd, float rms_coef, int ns_steps, float a, float b,
                       float c, float eps, int nesterov, void* ws, size_t ws_bytes, mc_stream_t stream) {
    return muon_impl(true, w, g, m, nullptr, nullptr, rows, cols, count, lr, mu, wd, rms_coef, ns_steps, a, b, c,
                     eps, nesterov, ws, ws_bytes, (cudaStream_t)stream);
}

// ===========================================================================
// data-parallel exchange helpers (Distributed Muon, S_max over ranks)
// ===========================================================================

mc_status mc_smax_to_keys(const float* s_max, int* keys, int n, mc_stream_t stream) {
    if (n < 0 || (n > 0 && (!s_max || !keys))) return MC_ERR_INVALID_ARG;
    if (n > 0 && (!aligned4(s_max) || !aligned4(keys))) return MC_ERR_INVALID_ARG;
    MC_CUDA(launch_smax_keys(s_max, keys, nullptr, nullptr, n, (cudaStream_t)stream));
    return MC_OK;
}

mc_status mc_smax_from_keys(const int* keys, float* s_max, int n, mc_stream_t stream) {
    if (n < 0 || (n > 0 && (!s_max || !keys))) return MC_ERR_INVALID_ARG;
    if (n > 0 && (!aligned4(s_max) || !aligned4(keys))) return MC_ERR_INVALID_ARG;
    MC_CUDA(launch_smax_keys(nullptr, nullptr, keys, s_max, n, (cudaStream_t)stream));
    return MC_OK;
}

mc_status mc_muon_momentum(float* m, const float* g, float* u, size_t n, float mu, float grad_scale, int nesterov,
                           mc_stream_t stream) {
    if (n == 0) return MC_OK;
    if (!m || !g || (nesterov && !u)) return MC_ERR_INVALID_ARG;
    if (n > (size_t)INT64_MAX / 4) return MC_ERR_INVALID_ARG;
    if (!aligned4(m) || !aligned4(g) || (u && !aligned4(u))) return MC_ERR_INVALID_ARG;
    if ((const float*)m == g || u == m || (const float*)u == g) return MC_ERR_INVALID_ARG;
    MC_CUDA(launch_momentum_flat(m, g, u, (long long)n, mu, grad_scale, nesterov ? 1 : 0, (cudaStream_t)stream));
    return MC_OK;
}

mc_status mc_muon_apply(float* w, const float* o, size_t n, int rows, int cols, float lr, float rms_coef, float wd,
                        mc_stream_t stream) {
    if (n == 0) return MC_OK;
    if (!w || !o || rows <= 0 || cols <= 0 || (const float*)w == o) return MC_ERR_INVALID_ARG;
    if (n > (size_t)INT64_MAX / 4) return MC_ERR_INVALID_ARG;
    if (!aligned4(w) || !aligned4(o)) return MC_ERR_INVALID_ARG;
    // the RMS scale exactly as the whole-matrix update forms it
    const float rms = rms_coef * sqrtf((float)std::max(rows, cols));
    MC_CUDA(launch_update_flat(w, o, (long long)n, lr, rms, wd, (cudaStream_t)stream));
    return MC_OK;
}

// ===========================================================================
// tensor-core GEMM
// ===========================================================================

mc_status mc_gemm_bf16(const void* a, const void* b, void* c, mc_dtype c_type, int M, int N, int K, int batch,
                       int b_kmajor, mc_stream_t stream) {
    if (!a || !b || !c || M <= 0 || N <= 0 || K <= 0 || batch <= 0) return MC_ERR_INVALID_ARG;
    if (c_type != MC_F32 && c_type != MC_BF16) return MC_ERR_INVALID_ARG;
    if (K % 8 || (!b_kmajor && N % 8)) return MC_ERR_UNSUPPORTED;
    if (!aligned16(a) || !aligned16(b) || !aligned16(c)) return MC_ERR_INVALID_ARG;
    GemmParams P;
    memset(&P, 0, sizeof(P));
    P.nprob = 1;
    P.tile_m = kPairTileM;
    GemmProblem& q = P.p[0];
    const uint64_t m = M, n = N, k = K, z = batch;
    if (!make_tmap_3d(&q.tmA, a, k, m, z, k, m * k, kBK, kBM, 0)) return MC_ERR_INVALID_ARG;
    if (b_kmajor) {
        // a CTA of a pair loads half of the B tile's rows
        const uint32_t brows = P.tile_m == kBM ? kBN : kBN / 2;
        if (!make_tmap_3d(&q.tmB, b, k, n, z, k, n * k, kBK, brows, 0)) return MC_ERR_INVALID_ARG;
    } else {
        if (!make_tmap_3d(&q.tmB, b, n, k, z, n, k * n, 64, kStageKPair, 0)) return MC_ERR_INVALID_ARG;
        q.b_mn = 1;
    }
    q.M = M;
    q.N = N;
    q.K = K;
    q.batch = batch;
    q.out_kind = c_type == MC_F32 ? kOutF32 : kOutBF16;
    q.out = c;
    q.out_ld = N;
    q.out_bstride = (long long)M * N;
    q.alpha = 1.f;
    q.vec_ok = c_type == MC_F32 ? (N % 4 == 0) : (N % 8 == 0);
    if (c_type == MC_BF16 && q.vec_ok)
        q.bulk_st = make_tmap_3d(&q.tmC, c, n, m, z, n, m * n, 64, 32, 0);
    finalize_gemm_params(P);
    MC_CUDA(launch_gemm(P, (cudaStream_t)stream, "gemm"));
    return MC_OK;
}

}  // extern "C"
