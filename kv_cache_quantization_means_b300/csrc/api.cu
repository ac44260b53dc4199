// C ABI of the KV-cache codec: host-side validation, workspace carving and
// launch sequencing.  Declarations and contracts: include/qvg.h.
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include <cmath>

#include "attn.h"
#include "common.cuh"
#include "kernels.h"

namespace {

thread_local char g_err[512] = "";

qvg_status fail(qvg_status st, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return st;
}

qvg_status ok() {
    g_err[0] = '\0';
    return QVG_OK;
}

qvg_status cuda_status(cudaError_t e, const char* what) {
    if (e == cudaSuccess) return ok();
    return fail(QVG_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

constexpr int kMaxChunks = 4096;   // chunk table is staged in shared memory by the decoder

qvg_status check_config(const qvg_config* c, bool need_clusters) {
    if (!c) return fail(QVG_ERR_INVALID_ARG, "config is NULL");
    if (c->num_heads < 1) return fail(QVG_ERR_INVALID_ARG, "num_heads must be >= 1");
    if (c->bits != 2 && c->bits != 4) return fail(QVG_ERR_UNSUPPORTED, "bits must be 2 or 4 (got %d)", c->bits);
    const int D = c->head_dim, G = c->group_size;
    if (D != 32 && D != 64 && D != 128 && D != 256)
        return fail(QVG_ERR_UNSUPPORTED, "head_dim must be 32, 64, 128 or 256 (got %d)", D);
    if (G != 16 && G != 32 && G != 64 && G != 128)
        return fail(QVG_ERR_UNSUPPORTED, "group_size must be 16, 32, 64 or 128 (got %d)", G);
    if (G > D || D % G) return fail(QVG_ERR_INVALID_ARG, "group_size %d must divide head_dim %d", G, D);
    if (c->num_stages < 1 || c->num_stages > qvg::kMaxStages)
        return fail(QVG_ERR_UNSUPPORTED, "num_stages must be in 1..%d", qvg::kMaxStages);
    if (c->num_clusters < 0 || c->num_clusters > qvg::kMaxClusters)
        return fail(QVG_ERR_UNSUPPORTED, "num_clusters must be in 0..%d", qvg::kMaxClusters);
    if (c->num_clusters > 0 && D > 128)
        return fail(QVG_ERR_UNSUPPORTED, "k-means smoothing supports head_dim <= 128");
    if (need_clusters && c->num_clusters < 1)
        return fail(QVG_ERR_INVALID_ARG, "this call needs num_clusters >= 1");
    return QVG_OK;
}

qvg_status check_input(const qvg_config* c, const void* x, int64_t n, int64_t hs, int64_t ts,
                       const char* name) {
    if (n < 0) return fail(QVG_ERR_INVALID_ARG, "%s: negative token count", name);
    if (n == 0) return QVG_OK;
    if (!x) return fail(QVG_ERR_INVALID_ARG, "%s is NULL", name);
    if (!aligned16(x)) return fail(QVG_ERR_INVALID_ARG, "%s must be 16-byte aligned", name);
    if (hs % 8 || ts % 8) return fail(QVG_ERR_INVALID_ARG, "%s strides must be multiples of 8 elements", name);
    if (ts < c->head_dim && c->num_heads > 0 && hs < c->head_dim)
        return fail(QVG_ERR_INVALID_ARG, "%s strides overlap rows", name);
    if (hs < 0 || ts < 0) return fail(QVG_ERR_INVALID_ARG, "%s strides must be non-negative", name);
    return QVG_OK;
}

qvg_status check_rows(int64_t cap, int64_t off, int64_t n) {
    if (cap < 0 || off < 0 || n < 0) return fail(QVG_ERR_INVALID_ARG, "negative capacity/offset/count");
    if (off + n > cap)
        return fail(QVG_ERR_CAPACITY, "rows [%lld, %lld) exceed capacity %lld", (long long)off,
                    (long long)(off + n), (long long)cap);
    return QVG_OK;
}

size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }

struct FitWorkspace {
    unsigned long long* stats;  // [4]
    float* xnorm;       // [H][N] ||x||^2 per token, shared by a fit's assign steps
    long long* ksum;    // [H][C][3][D] exact window sums of each cluster's members
    int* kcount;        // [H][C]
    int* kbig;          // [H][C]
    int* chg_tok;       // [H][chg_stride] ids changed by the last assign
    uint16_t* chg_on;   // [H][chg_stride]
    int2* chg_parts;    // [H][kChgParts]
    int64_t chg_stride; // head stride of chg_tok / chg_on
    size_t bytes;
};

FitWorkspace carve(const qvg_config* c, int64_t n, void* base) {
    const size_t H = c->num_heads, C = c->num_clusters > 0 ? c->num_clusters : 1, D = c->head_dim;
    const size_t N = (size_t)(n > 0 ? n : 1);
    FitWorkspace w{};
    size_t o = 0;
    auto take = [&](size_t bytes) {
        size_t at = o;
        o += align256(bytes);
        return base ? (void*)((char*)base + at) : nullptr;
    };
    w.stats = (unsigned long long*)take(sizeof(unsigned long long) * 4);
    w.xnorm = (float*)take(sizeof(float) * H * N);
    w.ksum = (long long*)take(sizeof(long long) * H * C * 3 * D);
    w.kcount = (int*)take(sizeof(int) * H * C);
    w.kbig = (int*)take(sizeof(int) * H * C);
    w.chg_stride = (int64_t)((N + 7) / 8 * 8);
    w.chg_tok = (int*)take(sizeof(int) * H * (size_t)w.chg_stride);
    w.chg_on = (uint16_t*)take(sizeof(uint16_t) * H * (size_t)w.chg_stride);
    w.chg_parts = (int2*)take(sizeof(int2) * H * qvg::kChgParts);
    w.bytes = o;
    return w;
}

qvg_status check_workspace(const qvg_config* c, int64_t n, void* ws, size_t ws_bytes, FitWorkspace* out) {
    FitWorkspace need = carve(c, n, nullptr);
    if (!ws) return fail(QVG_ERR_INVALID_ARG, "workspace is NULL (need %zu bytes)", need.bytes);
    if (((uintptr_t)ws & 255u) != 0) return fail(QVG_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
    if (ws_bytes < need.bytes)
        return fail(QVG_ERR_INVALID_ARG, "workspace too small: %zu < %zu bytes", ws_bytes, need.bytes);
    *out = carve(c, n, ws);
    return QVG_OK;
}

// Workspace of the cross-layer calls: the low-rank projection (fp32 [N][64])
// or the tensor-core path's scratch, whichever is larger.
size_t coral_ws_bytes(const qvg_config* c, int64_t n_tokens) {
    const size_t lr = align256(sizeof(float) * 64 * (size_t)(n_tokens > 0 ? n_tokens : 1));
    const size_t tc = qvg::coral_tc_scratch_bytes(c->num_heads, n_tokens);
    return lr > tc ? lr : tc;
}

// coral_fit_block: the tensor-core scratch (t, W^T, [U|U], error word), then
// the fp32 partial Gram sums.
size_t coral_fit_ws_bytes(const qvg_config* c, int64_t n_tokens) {
    return qvg::coral_tc_scratch_bytes(c->num_heads, n_tokens) + align256(qvg::coral_fit_part_bytes(c->num_heads, n_tokens));
}

qvg::AssignArgs assign_args(const qvg_config* c, const qvg_bf16* x, int64_t n, int64_t hs, int64_t ts,
                            const qvg_bf16* cent, uint8_t* ids, int64_t cap, int64_t off, int* counts,
                            unsigned long long* stats) {
    qvg::AssignArgs a;
    a.x = x; a.head_stride = hs; a.token_stride = ts; a.n_tokens = n;
    a.cent = cent; a.C = c->num_clusters;
    a.ids = ids; a.cap = cap; a.tok_offset = off;
    a.counts = counts; a.stats = stats;
    a.err = stats ? reinterpret_cast<uint32_t*>(stats + 3) : nullptr;
    a.xnorm = nullptr;
    a.xnorm_mode = qvg::kNormCompute;
    a.chg_tok = nullptr; a.chg_on = nullptr; a.chg_parts = nullptr; a.chg_stride = 0;
    return a;
}

qvg::UpdateArgs update_args(const qvg_config* c, const qvg_bf16* x, int64_t n, int64_t hs, int64_t ts,
                            const uint8_t* ids, int64_t cap, int64_t off, const FitWorkspace& w, qvg_bf16* cent) {
    qvg::UpdateArgs u;
    u.x = x; u.head_stride = hs; u.token_stride = ts; u.n_tokens = n;
    u.ids = ids; u.cap = cap; u.tok_offset = off;
    u.H = c->num_heads; u.C = c->num_clusters;
    u.group_log2 = -1;
    u.cent = cent;
    u.ksum = w.ksum; u.kcount = w.kcount; u.kbig = w.kbig;
    u.chg_tok = w.chg_tok; u.chg_on = w.chg_on; u.chg_parts = w.chg_parts; u.chg_stride = w.chg_stride;
    u.mode = qvg::kUpdFull;
    return u;
}

// T Lloyd iterations (init already in `cent`).  The first update sums every
// cluster; each later one applies only the ids that the assign before it
// changed, to the exact sums the previous update stored in the workspace.
qvg_status lloyd(const qvg_config* c, const qvg_bf16* x, int64_t n, int64_t hs, int64_t ts,
                 qvg_bf16* cent, uint8_t* ids, int64_t cap, int64_t off, const FitWorkspace& w,
                 cudaStream_t s, bool clear_stats = true) {
    cudaError_t e = cudaSuccess;
    if (clear_stats && (e = cudaMemsetAsync(w.stats, 0, sizeof(unsigned long long) * 4, s)) != cudaSuccess)
        return cuda_status(e, "memset");
    bool have_sums = false;    // the workspace holds the exact sums of the current ids
    for (int t = 0; t < c->lloyd_iters; ++t) {
        // x is the same in every step: the first assign stores ||x||^2 per
        // token, the later ones read it
        qvg::AssignArgs aa = assign_args(c, x, n, hs, ts, cent, ids, cap, off, nullptr, w.stats);
        aa.xnorm = w.xnorm;
        aa.xnorm_mode = t == 0 ? qvg::kNormStore : qvg::kNormLoad;
        if (have_sums) {
            if ((e = cudaMemsetAsync(w.chg_parts, 0, sizeof(int2) * c->num_heads * qvg::kChgParts, s)) != cudaSuccess)
                return cuda_status(e, "memset");
            aa.chg_tok = w.chg_tok; aa.chg_on = w.chg_on; aa.chg_parts = w.chg_parts; aa.chg_stride = w.chg_stride;
        }
        bool recorded = false;
        e = qvg::launch_assign(c->head_dim, c->num_heads, aa, s, &recorded);
        if (e != cudaSuccess) return cuda_status(e, "assign launch");
        qvg::UpdateArgs u = update_args(c, x, n, hs, ts, ids, cap, off, w, cent);
        u.mode = have_sums && recorded ? qvg::kUpdIncremental : qvg::kUpdFull;
        e = qvg::launch_update(c->head_dim, u, s);
        if (e != cudaSuccess) return cuda_status(e, "update launch");
        have_sums = true;
    }
    return ok();
}

}  // namespace

extern "C" {

const char* qvg_last_error(void) { return g_err; }

const char* qvg_version(void) { return "qvg-b300 0.1 (sm_103a)"; }

qvg_status qvg_encoded_bytes(const qvg_config* cfg, int64_t capacity, int32_t n_versions, size_t* codes_bytes,
                             size_t* meta_bytes, size_t* ids_bytes, size_t* centroid_bytes) {
    qvg_status st = check_config(cfg, false);
    if (st) return st;
    if (capacity < 0 || n_versions < 0) return fail(QVG_ERR_INVALID_ARG, "negative capacity or versions");
    const size_t S = cfg->num_stages, H = cfg->num_heads, D = cfg->head_dim, G = cfg->group_size,
                 C = cfg->num_clusters, N = (size_t)capacity;
    if (codes_bytes) *codes_bytes = S * H * N * (D * (size_t)cfg->bits / 32) * 4;
    if (meta_bytes) *meta_bytes = S * H * N * (D / G) * 4;
    if (ids_bytes) *ids_bytes = C ? H * N : 0;
    if (centroid_bytes) *centroid_bytes = C ? (size_t)n_versions * H * C * D * 2 : 0;
    return ok();
}

qvg_status qvg_workspace_bytes(const qvg_config* cfg, int64_t n_tokens, size_t* bytes) {
    qvg_status st = check_config(cfg, false);
    if (st) return st;
    if (!bytes || n_tokens < 0) return fail(QVG_ERR_INVALID_ARG, "bad arguments");
    size_t b = carve(cfg, n_tokens, nullptr).bytes;
    if (cfg->num_clusters == 0) {
        size_t coral = coral_ws_bytes(cfg, n_tokens);
        if (coral > b) b = coral;
        if (cfg->head_dim == 128) {
            const size_t fit = coral_fit_ws_bytes(cfg, n_tokens);
            if (fit > b) b = fit;
        }
    }
    *bytes = b;
    return ok();
}

qvg_status qvg_fit_stats(const qvg_config* cfg, int64_t n_tokens, const void* workspace, size_t workspace_bytes,
                         uint64_t* out, qvg_stream stream) {
    qvg_status st = check_config(cfg, false);
    if (st) return st;
    if (!out) return fail(QVG_ERR_INVALID_ARG, "out is NULL");
    if (n_tokens < 0) return fail(QVG_ERR_INVALID_ARG, "negative token count");
    if (cfg->num_clusters == 0) {
        // cross-layer config: only the error word of the tensor-core path
        const size_t tc = qvg::coral_tc_scratch_bytes(cfg->num_heads, n_tokens);
        out[0] = out[1] = out[2] = out[3] = 0;
        if (!workspace || workspace_bytes < tc) return ok();
        uint32_t w = 0;
        cudaStream_t s = (cudaStream_t)stream;
        cudaError_t e = cudaMemcpyAsync(&w, static_cast<const char*>(workspace) + tc - 256, sizeof(w),
                                        cudaMemcpyDeviceToHost, s);
        if (e == cudaSuccess) e = cudaStreamSynchronize(s);
        if (e != cudaSuccess) return cuda_status(e, "stats copy");
        out[3] = w;
        if (w) return fail(QVG_ERR_TIMEOUT, "a kernel gave up a bounded wait (error word 0x%08x)", w);
        return ok();
    }
    FitWorkspace w;
    if ((st = check_workspace(cfg, n_tokens, const_cast<void*>(workspace), workspace_bytes, &w))) return st;
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e = cudaMemcpyAsync(out, w.stats, sizeof(unsigned long long) * 4, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_status(e, "stats copy");
    out[3] &= 0xFFFFFFFFull;
    if (out[3]) return fail(QVG_ERR_TIMEOUT, "a kernel gave up a bounded wait (error word 0x%08x)", (unsigned)out[3]);
    return ok();
}

qvg_status qvg_device_error(uint32_t* out, int32_t clear, qvg_stream stream) {
    if (!out) return fail(QVG_ERR_INVALID_ARG, "out is NULL");
    qvg_status st = cuda_status(qvg::read_codec_error(out, clear != 0, (cudaStream_t)stream), "device error word");
    if (st) return st;
    if (*out) return fail(QVG_ERR_TIMEOUT, "a kernel gave up a bounded wait (error word 0x%08x)", *out);
    return ok();
}

qvg_status qvg_debug_set_wait(uint64_t wait_limit_ns, uint32_t flags, qvg_stream stream) {
    if (flags > 1u) return fail(QVG_ERR_INVALID_ARG, "unknown debug flags 0x%x", flags);
    const unsigned long long limit = wait_limit_ns ? (unsigned long long)wait_limit_ns : 2000000000ull;
    return cuda_status(qvg::set_codec_debug(limit, flags, (cudaStream_t)stream), "debug settings");
}

qvg_status qvg_fit_centroids(const qvg_config* cfg, const qvg_bf16* x, int64_t n_tokens, int64_t head_stride,
                             int64_t token_stride, const qvg_bf16* warm_start, qvg_bf16* centroids, uint8_t* ids,
                             int64_t capacity, int64_t tok_offset, void* workspace, size_t workspace_bytes,
                             qvg_stream stream) {
    qvg_status st = check_config(cfg, true);
    if (st) return st;
    if (cfg->lloyd_iters < 1) return fail(QVG_ERR_INVALID_ARG, "lloyd_iters must be >= 1");
    if (n_tokens < 1) return fail(QVG_ERR_INVALID_ARG, "fit needs n_tokens >= 1");
    if ((st = check_input(cfg, x, n_tokens, head_stride, token_stride, "x"))) return st;
    if (!centroids || !aligned16(centroids)) return fail(QVG_ERR_INVALID_ARG, "centroids NULL or unaligned");
    if (warm_start && !aligned16(warm_start)) return fail(QVG_ERR_INVALID_ARG, "warm_start unaligned");
    if (!ids) return fail(QVG_ERR_INVALID_ARG, "ids is NULL");
    if ((st = check_rows(capacity, tok_offset, n_tokens))) return st;
    FitWorkspace w;
    if ((st = check_workspace(cfg, n_tokens, workspace, workspace_bytes, &w))) return st;
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e = qvg::launch_kmeans_init(cfg->head_dim, x, head_stride, token_stride, n_tokens, warm_start,
                                            cfg->num_heads, cfg->num_clusters, centroids, s);
    if (e != cudaSuccess) return cuda_status(e, "init launch");
    return lloyd(cfg, x, n_tokens, head_stride, token_stride, centroids, ids, capacity, tok_offset, w, s);
}

qvg_status qvg_assign(const qvg_config* cfg, const qvg_bf16* x, int64_t n_tokens, int64_t head_stride,
                      int64_t token_stride, const qvg_bf16* centroids, uint8_t* ids, int64_t capacity,
                      int64_t tok_offset, void* workspace, size_t workspace_bytes, qvg_stream stream) {
    qvg_status st = check_config(cfg, true);
    if (st) return st;
    if ((st = check_input(cfg, x, n_tokens, head_stride, token_stride, "x"))) return st;
    if (!centroids || !aligned16(centroids)) return fail(QVG_ERR_INVALID_ARG, "centroids NULL or unaligned");
    if (!ids) return fail(QVG_ERR_INVALID_ARG, "ids is NULL");
    if ((st = check_rows(capacity, tok_offset, n_tokens))) return st;
    FitWorkspace w;
    if ((st = check_workspace(cfg, n_tokens, workspace, workspace_bytes, &w))) return st;
    cudaError_t e = cudaMemsetAsync(w.stats, 0, sizeof(unsigned long long) * 4, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_status(e, "memset");
    e = qvg::launch_assign(
        cfg->head_dim, cfg->num_heads,
        assign_args(cfg, x, n_tokens, head_stride, token_stride, centroids, ids, capacity, tok_offset, nullptr,
                    w.stats),
        (cudaStream_t)stream);
    return cuda_status(e, "assign launch");
}

qvg_status qvg_update(const qvg_config* cfg, const qvg_bf16* x, int64_t n_tokens, int64_t head_stride,
                      int64_t token_stride, const uint8_t* ids, int64_t capacity, int64_t tok_offset,
                      qvg_bf16* centroids, void* workspace, size_t workspace_bytes, qvg_stream stream) {
    qvg_status st = check_config(cfg, true);
    if (st) return st;
    if ((st = check_input(cfg, x, n_tokens, head_stride, token_stride, "x"))) return st;
    if (!centroids || !aligned16(centroids)) return fail(QVG_ERR_INVALID_ARG, "centroids NULL or unaligned");
    if (!ids) return fail(QVG_ERR_INVALID_ARG, "ids is NULL");
    if ((st = check_rows(capacity, tok_offset, n_tokens))) return st;
    FitWorkspace w;
    if ((st = check_workspace(cfg, n_tokens, workspace, workspace_bytes, &w))) return st;
    cudaStream_t s = (cudaStream_t)stream;
    qvg::UpdateArgs u = update_args(cfg, x, n_tokens, head_stride, token_stride, ids, capacity, tok_offset, w, centroids);
    cudaError_t e = qvg::launch_update(cfg->head_dim, u, s);
    return cuda_status(e, "update launch");
}

qvg_status qvg_encode(const qvg_config* cfg, const qvg_bf16* x, int64_t n_tokens, int64_t head_stride,
                      int64_t token_stride, const qvg_bf16* centroids, int32_t assign, uint32_t* codes, uint32_t* meta,
                      uint8_t* ids, int64_t capacity, int64_t tok_offset, void* workspace, size_t workspace_bytes,
                      qvg_stream stream) {
    qvg_status st = check_config(cfg, false);
    if (st) return st;
    if ((st = check_input(cfg, x, n_tokens, head_stride, token_stride, "x"))) return st;
    if (!codes || !meta) return fail(QVG_ERR_INVALID_ARG, "codes/meta is NULL");
    if (!aligned16(codes) || !aligned16(meta)) return fail(QVG_ERR_INVALID_ARG, "codes/meta must be 16-byte aligned");
    if ((st = check_rows(capacity, tok_offset, n_tokens))) return st;
    cudaStream_t s = (cudaStream_t)stream;
    const int C = cfg->num_clusters;
    if (C > 0) {
        if (!centroids || !aligned16(centroids)) return fail(QVG_ERR_INVALID_ARG, "centroids NULL or unaligned");
        if (!ids) return fail(QVG_ERR_INVALID_ARG, "ids is NULL");
        if (assign) {
            FitWorkspace w;
            if ((st = check_workspace(cfg, n_tokens, workspace, workspace_bytes, &w))) return st;
            cudaError_t e = cudaMemsetAsync(w.stats, 0, sizeof(unsigned long long) * 4, s);
            if (e != cudaSuccess) return cuda_status(e, "memset");
            e = qvg::launch_assign(cfg->head_dim, cfg->num_heads,
                                               assign_args(cfg, x, n_tokens, head_stride, token_stride, centroids,
                                                           ids, capacity, tok_offset, nullptr, w.stats),
                                               s);
            if (e != cudaSuccess) return cuda_status(e, "assign launch");
        }
    }
    qvg::EncodeArgs a;
    a.x = x; a.head_stride = head_stride; a.token_stride = token_stride; a.n_tokens = n_tokens;
    a.cent = C > 0 ? centroids : nullptr;
    a.ids = C > 0 ? ids : nullptr;
    a.codes = codes; a.meta = meta; a.cap = capacity; a.tok_offset = tok_offset;
    a.H = cfg->num_heads; a.C = C; a.S = cfg->num_stages; a.bits = cfg->bits;
    return cuda_status(qvg::launch_encode(cfg->head_dim, cfg->group_size, a, s), "encode launch");
}

static qvg_status decode_impl(const qvg_config* cfg, const uint32_t* codes, const uint32_t* meta, const uint8_t* ids,
                              const qvg_bf16* centroids, const int64_t* chunk_offset, const int32_t* chunk_version,
                              int n_chunks, int64_t capacity, int64_t tok_begin, int64_t tok_end, qvg_bf16* out,
                              int64_t ohs, int64_t ots, cudaStream_t s) {
    if (tok_begin < 0 || tok_end < tok_begin || tok_end > capacity)
        return fail(QVG_ERR_INVALID_ARG, "token range [%lld, %lld) outside [0, %lld)", (long long)tok_begin,
                    (long long)tok_end, (long long)capacity);
    if (tok_end == tok_begin) return ok();
    if (!codes || !meta || !out) return fail(QVG_ERR_INVALID_ARG, "codes/meta/out is NULL");
    if (!aligned16(codes) || !aligned16(meta) || !aligned16(out))
        return fail(QVG_ERR_INVALID_ARG, "codes/meta/out must be 16-byte aligned");
    if (ohs % 8 || ots % 8 || ohs < 0 || ots < 0) return fail(QVG_ERR_INVALID_ARG, "out strides must be multiples of 8");
    if (cfg->num_clusters > 0 && (!ids || !centroids || !aligned16(centroids)))
        return fail(QVG_ERR_INVALID_ARG, "ids/centroids missing");
    qvg::DecodeArgs a;
    a.codes = codes; a.meta = meta; a.ids = ids; a.cent = centroids;
    a.chunk_offset = chunk_offset; a.chunk_version = chunk_version; a.n_chunks = n_chunks;
    a.cap = capacity; a.tok_begin = tok_begin; a.tok_end = tok_end;
    a.out = out; a.out_head_stride = ohs; a.out_token_stride = ots;
    a.H = cfg->num_heads; a.C = cfg->num_clusters; a.S = cfg->num_stages; a.bits = cfg->bits;
    return cuda_status(qvg::launch_decode(cfg->head_dim, cfg->group_size, a, s), "decode launch");
}

qvg_status qvg_decode(const qvg_config* cfg, const uint32_t* codes, const uint32_t* meta, const uint8_t* ids,
                      const qvg_bf16* centroids, int64_t capacity, int64_t tok_begin, int64_t tok_end, qvg_bf16* out,
                      int64_t out_head_stride, int64_t out_token_stride, qvg_stream stream) {
    qvg_status st = check_config(cfg, false);
    if (st) return st;
    return decode_impl(cfg, codes, meta, ids, centroids, nullptr, nullptr, 0, capacity, tok_begin, tok_end, out,
                       out_head_stride, out_token_stride, (cudaStream_t)stream);
}

qvg_status qvg_compress_host(const qvg_config* cfg, const qvg_bf16* x_host, qvg_bf16* x_dev, int64_t n_tokens,
                             int64_t head_stride, int64_t token_stride, const qvg_bf16* warm_start,
                             qvg_bf16* centroids, uint8_t* ids, uint32_t* codes, uint32_t* meta, qvg_bf16* out_dev,
                             void* host_out, size_t host_out_bytes, void* workspace, size_t workspace_bytes,
                             qvg_stream stream) {
    qvg_status st = check_config(cfg, false);
    if (st) return st;
    if (n_tokens < 1) return fail(QVG_ERR_INVALID_ARG, "n_tokens must be >= 1");
    if (!x_host || !host_out) return fail(QVG_ERR_INVALID_ARG, "host buffers are NULL");
    if ((st = check_input(cfg, x_dev, n_tokens, head_stride, token_stride, "x_dev"))) return st;
    const int64_t span = (n_tokens - 1) * token_stride + (int64_t)(cfg->num_heads - 1) * head_stride + cfg->head_dim;
    size_t cb = 0, mb = 0, ib = 0, xb = 0;
    if ((st = qvg_encoded_bytes(cfg, n_tokens, 1, &cb, &mb, &ib, &xb))) return st;
    if (host_out_bytes < cb + mb + ib + xb)
        return fail(QVG_ERR_INVALID_ARG, "host_out too small: %zu < %zu bytes", host_out_bytes, cb + mb + ib + xb);
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e = cudaMemcpyAsync(x_dev, x_host, (size_t)span * sizeof(qvg_bf16), cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return cuda_status(e, "host-to-device copy");
    if (cfg->num_clusters > 0) {
        st = qvg_fit_centroids(cfg, x_dev, n_tokens, head_stride, token_stride, warm_start, centroids, ids, n_tokens,
                               0, workspace, workspace_bytes, stream);
        if (st) return st;
    }
    st = qvg_encode(cfg, x_dev, n_tokens, head_stride, token_stride, centroids, 0, codes, meta, ids, n_tokens, 0,
                    workspace, workspace_bytes, stream);
    if (st) return st;
    if (out_dev) {
        st = qvg_decode(cfg, codes, meta, ids, centroids, n_tokens, 0, n_tokens, out_dev, head_stride, token_stride,
                        stream);
        if (st) return st;
    }
    char* h = static_cast<char*>(host_out);
    const void* src[4] = {codes, meta, ids, centroids};
    const size_t nb[4] = {cb, mb, ib, xb};
    for (int k = 0; k < 4; ++k) {
        if (!nb[k]) continue;
        if ((e = cudaMemcpyAsync(h, src[k], nb[k], cudaMemcpyDeviceToHost, s)) != cudaSuccess)
            return cuda_status(e, "device-to-host copy");
        h += nb[k];
    }
    return ok();
}

qvg_status qvg_append_chunk(const qvg_config* cfg, qvg_cache* cache, const qvg_bf16* x, int64_t n_new,
                            int64_t head_stride, int64_t token_stride, int32_t refit, void* workspace,
                            size_t workspace_bytes, qvg_stream stream) {
    qvg_status st = check_config(cfg, true);
    if (st) return st;
    if (!cache) return fail(QVG_ERR_INVALID_ARG, "cache is NULL");
    if (n_new < 1) return fail(QVG_ERR_INVALID_ARG, "append needs n_new >= 1");
    if (!cache->codes || !cache->meta || !cache->ids || !cache->centroids || !cache->chunk_offset ||
        !cache->chunk_version)
        return fail(QVG_ERR_INVALID_ARG, "cache buffers missing");
    if ((st = check_input(cfg, x, n_new, head_stride, token_stride, "x"))) return st;
    if (cache->n_used < 0 || cache->n_chunks < 0 || cache->n_versions < 0)
        return fail(QVG_ERR_INVALID_ARG, "corrupt cache counters");
    if (cache->max_chunks > kMaxChunks)
        return fail(QVG_ERR_UNSUPPORTED, "max_chunks must be <= %d", kMaxChunks);
    if (cache->n_chunks >= cache->max_chunks) return fail(QVG_ERR_CAPACITY, "chunk table full (%d)", cache->max_chunks);
    if (refit && cache->n_versions >= cache->max_versions)
        return fail(QVG_ERR_CAPACITY, "centroid versions full (%d)", cache->max_versions);
    if (!refit && cache->n_versions == 0)
        return fail(QVG_ERR_INVALID_ARG, "first chunk must refit (no centroid table yet)");
    if ((st = check_rows(cache->capacity, cache->n_used, n_new))) return st;
    if (cfg->lloyd_iters < 1 && refit) return fail(QVG_ERR_INVALID_ARG, "lloyd_iters must be >= 1");
    FitWorkspace w;
    if ((st = check_workspace(cfg, n_new, workspace, workspace_bytes, &w))) return st;
    cudaStream_t s = (cudaStream_t)stream;
    const size_t table = (size_t)cfg->num_heads * cfg->num_clusters * cfg->head_dim;
    int version = cache->n_versions - 1;
    if (refit) {
        version = cache->n_versions;
        const qvg_bf16* warm = cache->n_versions ? cache->centroids + (size_t)(cache->n_versions - 1) * table : nullptr;
        qvg_bf16* dst = cache->centroids + (size_t)version * table;
        cudaError_t e = qvg::launch_kmeans_init(cfg->head_dim, x, head_stride, token_stride, n_new, warm,
                                                cfg->num_heads, cfg->num_clusters, dst, s);
        if (e != cudaSuccess) return cuda_status(e, "init launch");
        if ((st = lloyd(cfg, x, n_new, head_stride, token_stride, dst, cache->ids, cache->capacity, cache->n_used, w,
                        s)))
            return st;
    }
    st = qvg_encode(cfg, x, n_new, head_stride, token_stride, cache->centroids + (size_t)version * table,
                    refit ? 0 : 1, cache->codes, cache->meta, cache->ids, cache->capacity, cache->n_used, workspace,
                    workspace_bytes, stream);
    if (st) return st;
    cudaError_t e = qvg::launch_set_chunk(cache->chunk_offset, cache->chunk_version, cache->n_chunks, cache->n_used,
                                          cache->n_used + n_new, version, s);
    if (e != cudaSuccess) return cuda_status(e, "chunk table launch");
    cache->n_used += n_new;
    cache->n_chunks += 1;
    if (refit) cache->n_versions += 1;
    return ok();
}

qvg_status qvg_decode_cache(const qvg_config* cfg, const qvg_cache* cache, int64_t tok_begin, int64_t tok_end,
                            qvg_bf16* out, int64_t out_head_stride, int64_t out_token_stride, qvg_stream stream) {
    qvg_status st = check_config(cfg, true);
    if (st) return st;
    if (!cache) return fail(QVG_ERR_INVALID_ARG, "cache is NULL");
    if (tok_end > cache->n_used)
        return fail(QVG_ERR_INVALID_ARG, "tok_end %lld beyond the %lld encoded rows", (long long)tok_end,
                    (long long)cache->n_used);
    if (tok_end > tok_begin && cache->n_chunks < 1) return fail(QVG_ERR_INVALID_ARG, "cache holds no chunk");
    if (cache->n_chunks > kMaxChunks || cache->n_chunks > cache->max_chunks)
        return fail(QVG_ERR_INVALID_ARG, "corrupt chunk count %d", cache->n_chunks);
    return decode_impl(cfg, cache->codes, cache->meta, cache->ids, cache->centroids, cache->chunk_offset,
                       cache->chunk_version, cache->n_chunks, cache->capacity, tok_begin, tok_end, out,
                       out_head_stride, out_token_stride, (cudaStream_t)stream);
}

// Zeroes the error word of the tensor-core cross-layer path (the word sits at
// the end of its scratch) when the workspace is large enough for that path.
static void clear_coral_error(const qvg_config* cfg, int64_t n_tokens, void* ws, size_t ws_bytes, cudaStream_t s) {
    const size_t tc = qvg::coral_tc_scratch_bytes(cfg->num_heads, n_tokens);
    if (ws_bytes >= tc) cudaMemsetAsync(static_cast<char*>(ws) + tc - 256, 0, sizeof(uint32_t), s);
}

// A prepared layout (coral_prepare_predictor) is for the rank-32, D = 128
// tensor-core path and must be 256-byte aligned.
static qvg_status check_prepared(const qvg_config* cfg, const coral_predictor* pred) {
    if (!pred->prepared) return QVG_OK;
    if (pred->rank != 32 || cfg->head_dim != 128)
        return fail(QVG_ERR_UNSUPPORTED, "a prepared predictor layout needs rank 32 and head_dim 128");
    if (((uintptr_t)pred->prepared & 255u) != 0) return fail(QVG_ERR_INVALID_ARG, "prepared layout must be 256-byte aligned");
    return QVG_OK;
}

static qvg_status coral_common(const qvg_config* cfg, const coral_predictor* pred, const qvg_bf16* xhat_prev,
                               int64_t n_tokens, void* workspace, size_t workspace_bytes) {
    qvg_status st = check_config(cfg, false);
    if (st) return st;
    if (cfg->num_clusters != 0) return fail(QVG_ERR_INVALID_ARG, "cross-layer codec needs num_clusters == 0");
    if (cfg->bits != 2) return fail(QVG_ERR_UNSUPPORTED, "cross-layer codec uses 2-bit codes (got %d)", cfg->bits);
    if (cfg->head_dim != 64 && cfg->head_dim != 128)
        return fail(QVG_ERR_UNSUPPORTED, "cross-layer codec supports head_dim 64 or 128");
    if (n_tokens < 0) return fail(QVG_ERR_INVALID_ARG, "negative token count");
    if (xhat_prev) {
        if (!pred || !pred->B) return fail(QVG_ERR_INVALID_ARG, "predictor missing");
        if (pred->rank < 0 || pred->rank > 64 || pred->rank % 16)
            return fail(QVG_ERR_UNSUPPORTED, "rank must be a multiple of 16 in 0..64");
        if (pred->rank > 0 && (!pred->U || !pred->W)) return fail(QVG_ERR_INVALID_ARG, "U/W missing");
        if (!aligned16(xhat_prev) || !aligned16(pred->B) || (pred->rank && (!aligned16(pred->U) || !aligned16(pred->W))))
            return fail(QVG_ERR_INVALID_ARG, "predictor / xhat_prev must be 16-byte aligned");
        const size_t need = coral_ws_bytes(cfg, n_tokens);
        if (pred->rank > 0 && (!workspace || workspace_bytes < need))
            return fail(QVG_ERR_INVALID_ARG, "workspace too small: need %zu bytes", need);
        if ((st = check_prepared(cfg, pred))) return st;
    }
    return QVG_OK;
}

qvg_status coral_predict_encode(const qvg_config* cfg, const coral_predictor* pred, const qvg_bf16* xhat_prev,
                                const qvg_bf16* x_next, int64_t n_tokens, uint32_t* codes, uint32_t* meta,
                                qvg_bf16* xhat_next, float* pred_out, void* workspace, size_t workspace_bytes,
                                qvg_stream stream) {
    qvg_status st = coral_common(cfg, pred, xhat_prev, n_tokens, workspace, workspace_bytes);
    if (st) return st;
    if (n_tokens == 0) return ok();
    if (!x_next || !codes || !meta || !xhat_next) return fail(QVG_ERR_INVALID_ARG, "buffer is NULL");
    if (!aligned16(x_next) || !aligned16(codes) || !aligned16(meta) || !aligned16(xhat_next) ||
        !aligned16(pred_out))
        return fail(QVG_ERR_INVALID_ARG, "buffers must be 16-byte aligned");
    qvg::CoralArgs a{};
    a.xprev = xhat_prev; a.xnext = x_next;
    a.B = xhat_prev ? pred->B : nullptr; a.U = xhat_prev ? pred->U : nullptr; a.W = xhat_prev ? pred->W : nullptr;
    a.R = xhat_prev ? pred->rank : 0;
    a.prepared = xhat_prev ? pred->prepared : nullptr;
    a.n_tokens = n_tokens; a.H = cfg->num_heads; a.S = cfg->num_stages;
    a.codes = codes; a.meta = meta; a.xhat = xhat_next; a.pred_out = pred_out;
    a.lowrank = (float*)workspace;
    a.workspace = workspace;
    a.workspace_bytes = workspace_bytes;
    if (workspace) clear_coral_error(cfg, n_tokens, workspace, workspace_bytes, (cudaStream_t)stream);
    return cuda_status(qvg::launch_coral(cfg->head_dim, cfg->group_size, true, a, (cudaStream_t)stream),
                       "coral launch");
}

qvg_status coral_prepared_bytes(const qvg_config* cfg, int32_t rank, size_t* bytes) {
    qvg_status st = check_config(cfg, false);
    if (st) return st;
    if (!bytes) return fail(QVG_ERR_INVALID_ARG, "bytes is NULL");
    if (rank != 32 || cfg->head_dim != 128)
        return fail(QVG_ERR_UNSUPPORTED, "a prepared predictor layout needs rank 32 and head_dim 128");
    *bytes = qvg::coral_prepared_bytes(cfg->num_heads);
    return ok();
}

qvg_status coral_prepare_predictor(const qvg_config* cfg, const coral_predictor* pred, qvg_bf16* prepared,
                                   size_t prepared_bytes, qvg_stream stream) {
    qvg_status st = check_config(cfg, false);
    if (st) return st;
    if (!pred || !pred->U || !pred->W || !prepared) return fail(QVG_ERR_INVALID_ARG, "predictor or buffer is NULL");
    if (pred->rank != 32 || cfg->head_dim != 128)
        return fail(QVG_ERR_UNSUPPORTED, "a prepared predictor layout needs rank 32 and head_dim 128");
    if (!aligned16(pred->U) || !aligned16(pred->W)) return fail(QVG_ERR_INVALID_ARG, "U/W must be 16-byte aligned");
    if (((uintptr_t)prepared & 255u) != 0) return fail(QVG_ERR_INVALID_ARG, "prepared layout must be 256-byte aligned");
    const size_t need = qvg::coral_prepared_bytes(cfg->num_heads);
    if (prepared_bytes < need) return fail(QVG_ERR_INVALID_ARG, "prepared buffer too small: need %zu bytes", need);
    return cuda_status(qvg::launch_coral_prep(pred->W, pred->U, cfg->num_heads, prepared, (cudaStream_t)stream),
                       "prep launch");
}

qvg_status coral_fit_block(const qvg_config* cfg, const coral_predictor* pred, const qvg_bf16* xhat_prev,
                           const qvg_bf16* x_next, int64_t n_tokens, qvg_bf16* B_out, void* workspace,
                           size_t workspace_bytes, qvg_stream stream) {
    qvg_status st = check_config(cfg, false);
    if (st) return st;
    if (cfg->num_clusters != 0) return fail(QVG_ERR_INVALID_ARG, "cross-layer codec needs num_clusters == 0");
    if (cfg->head_dim != 128) return fail(QVG_ERR_UNSUPPORTED, "block refit supports head_dim 128");
    if (!pred || pred->rank != 32 || !pred->U || !pred->W)
        return fail(QVG_ERR_UNSUPPORTED, "block refit needs the rank-32 low-rank part (U, W)");
    if (n_tokens < 1) return fail(QVG_ERR_INVALID_ARG, "block refit needs n_tokens >= 1");
    if (!xhat_prev || !x_next || !B_out) return fail(QVG_ERR_INVALID_ARG, "buffer is NULL");
    if (!aligned16(xhat_prev) || !aligned16(x_next) || !aligned16(B_out) || !aligned16(pred->U) || !aligned16(pred->W))
        return fail(QVG_ERR_INVALID_ARG, "buffers must be 16-byte aligned");
    const size_t need = coral_fit_ws_bytes(cfg, n_tokens);
    if (!workspace || workspace_bytes < need) return fail(QVG_ERR_INVALID_ARG, "workspace too small: need %zu bytes", need);
    if (((uintptr_t)workspace & 255u) != 0) return fail(QVG_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
    cudaStream_t s = (cudaStream_t)stream;
    clear_coral_error(cfg, n_tokens, workspace, workspace_bytes, s);
    const size_t N = (size_t)n_tokens, HD = (size_t)cfg->num_heads * 128;
    const size_t tc = qvg::coral_tc_scratch_bytes(cfg->num_heads, n_tokens);
    uint8_t* base = static_cast<uint8_t*>(workspace);
    qvg::CoralTcScratch w;
    w.t2 = reinterpret_cast<uint16_t*>(base);
    w.wt = reinterpret_cast<uint16_t*>(base + align256(N * 64 * 2));
    w.ud = reinterpret_cast<uint16_t*>(base + align256(N * 64 * 2) + align256(32 * HD * 2));
    if (pred->prepared) qvg::use_prepared(pred->prepared, cfg->num_heads, w);
    w.err = reinterpret_cast<uint32_t*>(base + tc - 256);
    if ((st = check_prepared(cfg, pred))) return st;
    qvg::CoralArgs a{};
    a.xprev = xhat_prev; a.U = pred->U; a.W = pred->W; a.R = 32;
    a.prepared = pred->prepared;
    a.n_tokens = n_tokens; a.H = cfg->num_heads; a.S = cfg->num_stages;
    cudaError_t e = qvg::launch_coral_lowrank_tc(a, w, s);
    if (e != cudaSuccess) return cuda_status(e, "low-rank launch");
    e = qvg::launch_coral_fit(xhat_prev, x_next, w.t2, pred->U, n_tokens, cfg->num_heads,
                              reinterpret_cast<float*>(base + tc), B_out, s);
    return cuda_status(e, "block refit launch");
}

qvg_status coral_predict_decode(const qvg_config* cfg, const coral_predictor* pred, const qvg_bf16* xhat_prev,
                                int64_t n_tokens, const uint32_t* codes, const uint32_t* meta, qvg_bf16* xhat_next,
                                float* pred_out, void* workspace, size_t workspace_bytes, qvg_stream stream) {
    qvg_status st = coral_common(cfg, pred, xhat_prev, n_tokens, workspace, workspace_bytes);
    if (st) return st;
    if (n_tokens == 0) return ok();
    if (!codes || !meta || !xhat_next) return fail(QVG_ERR_INVALID_ARG, "buffer is NULL");
    if (!aligned16(codes) || !aligned16(meta) || !aligned16(xhat_next) || !aligned16(pred_out))
        return fail(QVG_ERR_INVALID_ARG, "buffers must be 16-byte aligned");
    qvg::CoralArgs a{};
    a.xprev = xhat_prev; a.xnext = nullptr;
    a.B = xhat_prev ? pred->B : nullptr; a.U = xhat_prev ? pred->U : nullptr; a.W = xhat_prev ? pred->W : nullptr;
    a.R = xhat_prev ? pred->rank : 0;
    a.prepared = xhat_prev ? pred->prepared : nullptr;
    a.n_tokens = n_tokens; a.H = cfg->num_heads; a.S = cfg->num_stages;
    a.codes = const_cast<uint32_t*>(codes); a.meta = const_cast<uint32_t*>(meta);
    a.xhat = xhat_next; a.pred_out = pred_out;
    a.lowrank = (float*)workspace;
    a.workspace = workspace;
    a.workspace_bytes = workspace_bytes;
    if (workspace) clear_coral_error(cfg, n_tokens, workspace, workspace_bytes, (cudaStream_t)stream);
    return cuda_status(qvg::launch_coral(cfg->head_dim, cfg->group_size, false, a, (cudaStream_t)stream),
                       "coral launch");
}

// ------------------------------------------- allocation-free Coral encode
//
// Same computation as coral_predict_encode, for callers that cannot hand the
// library a workspace: the low-rank projection t = xhat_prev W ([n_tokens]
// x [rank] floats, the only scratch this call needs) lives in a file-scope
// device array of fixed size that every GPU loading the library keeps until
// the process exits.  Its device address is looked up once per device.

}  // extern "C"

namespace {

constexpr size_t kStaticScratchFloats = (size_t)1 << 20;          // 4 MiB
constexpr int64_t kStaticMaxTokens = (int64_t)(kStaticScratchFloats / 64);   // 64 floats per token (rank <= 64)
constexpr int kMaxDevices = 64;

static __device__ __align__(256) float g_coral_scratch[kStaticScratchFloats];

std::mutex g_scratch_mu;
float* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_coral_scratch on the current device (looked up with
// that device current, once per device).
qvg_status static_scratch(float** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_status(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(QVG_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_coral_scratch);
        if (e != cudaSuccess) return cuda_status(e, "cudaGetSymbolAddress(scratch)");
        g_scratch_ptr[dev] = static_cast<float*>(p);
    }
    *out = g_scratch_ptr[dev];
    return QVG_OK;
}

}  // namespace

extern "C" {

qvg_status coral_predict_encode_static(const qvg_config* cfg, const coral_predictor* pred,
                                       const qvg_bf16* xhat_prev, const qvg_bf16* x_next, int64_t n_tokens,
                                       uint32_t* codes, uint32_t* meta, qvg_bf16* xhat_next, float* pred_out,
                                       qvg_stream stream) {
    if (n_tokens > kStaticMaxTokens)
        return fail(QVG_ERR_CAPACITY, "n_tokens %lld exceeds the %lld tokens the built-in scratch holds",
                    (long long)n_tokens, (long long)kStaticMaxTokens);
    if (cfg && cfg->num_heads > 0 && xhat_prev && n_tokens > 0 &&
        coral_ws_bytes(cfg, n_tokens) > kStaticScratchFloats * sizeof(float))
        return fail(QVG_ERR_CAPACITY, "%d heads x %lld tokens need %zu bytes of scratch; the built-in array holds %zu",
                    cfg->num_heads, (long long)n_tokens, coral_ws_bytes(cfg, n_tokens),
                    kStaticScratchFloats * sizeof(float));
    float* scratch = nullptr;
    qvg_status st = QVG_OK;
    if (n_tokens > 0 && xhat_prev) {
        if ((st = static_scratch(&scratch))) return st;
    }
    st = coral_common(cfg, pred, xhat_prev, n_tokens, scratch, kStaticScratchFloats * sizeof(float));
    if (st) return st;
    if (n_tokens == 0) return ok();
    if (!x_next || !codes || !meta || !xhat_next) return fail(QVG_ERR_INVALID_ARG, "buffer is NULL");
    if (!aligned16(x_next) || !aligned16(codes) || !aligned16(meta) || !aligned16(xhat_next) ||
        !aligned16(pred_out))
        return fail(QVG_ERR_INVALID_ARG, "buffers must be 16-byte aligned");
    qvg::CoralArgs a{};
    a.xprev = xhat_prev; a.xnext = x_next;
    a.B = xhat_prev ? pred->B : nullptr; a.U = xhat_prev ? pred->U : nullptr; a.W = xhat_prev ? pred->W : nullptr;
    a.R = xhat_prev ? pred->rank : 0;
    a.prepared = xhat_prev ? pred->prepared : nullptr;
    a.n_tokens = n_tokens; a.H = cfg->num_heads; a.S = cfg->num_stages;
    a.codes = codes; a.meta = meta; a.xhat = xhat_next; a.pred_out = pred_out;
    a.lowrank = scratch;
    a.workspace = scratch;
    a.workspace_bytes = kStaticScratchFloats * sizeof(float);
    // a tensor-core wait that runs out is recorded in the library's device
    // error word (qvg_device_error), the only word this call can report through
    a.err_out = qvg::codec_error_word();
    if (scratch && !a.err_out) return fail(QVG_ERR_CUDA, "device error word lookup failed");
    return cuda_status(qvg::launch_coral(cfg->head_dim, cfg->group_size, true, a, (cudaStream_t)stream),
                       "coral launch");
}

}  // extern "C"

// ------------------------------------------------------ Coral-KV + SAS hybrid
//
// Workspace: [k-means fit workspace][cross-layer workspace][prediction, fp32
// [N][H*D]][residual / decoded residual, bf16 [N][H*D]], each 256-byte aligned.

namespace {

struct SasLayout {
    size_t fit, coral, pred, res, total;
};

SasLayout sas_layout(const qvg_config* cfg, int64_t n_tokens) {
    SasLayout L;
    const size_t N = (size_t)(n_tokens > 0 ? n_tokens : 1), HD = (size_t)cfg->num_heads * cfg->head_dim;
    qvg_config cc = *cfg;
    cc.num_clusters = 0;
    L.fit = 0;
    L.coral = align256(carve(cfg, n_tokens, nullptr).bytes);
    L.pred = L.coral + align256(coral_ws_bytes(&cc, n_tokens));
    L.res = L.pred + align256(N * HD * sizeof(float));
    L.total = L.res + align256(N * HD * 2);
    return L;
}

qvg_status sas_check(const qvg_config* cfg, const coral_predictor* pred, const qvg_bf16* xhat_prev,
                     int64_t n_tokens, void* workspace, size_t workspace_bytes, SasLayout* L) {
    qvg_status st = check_config(cfg, true);
    if (st) return st;
    if (cfg->bits != 2) return fail(QVG_ERR_UNSUPPORTED, "cross-layer codec uses 2-bit codes (got %d)", cfg->bits);
    if (cfg->lloyd_iters < 1) return fail(QVG_ERR_INVALID_ARG, "lloyd_iters must be >= 1");
    if (n_tokens < 1) return fail(QVG_ERR_INVALID_ARG, "the hybrid needs n_tokens >= 1");
    *L = sas_layout(cfg, n_tokens);
    if (!workspace) return fail(QVG_ERR_INVALID_ARG, "workspace is NULL (need %zu bytes)", L->total);
    if (((uintptr_t)workspace & 255u) != 0) return fail(QVG_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
    if (workspace_bytes < L->total)
        return fail(QVG_ERR_INVALID_ARG, "workspace too small: %zu < %zu bytes", workspace_bytes, L->total);
    qvg_config cc = *cfg;
    cc.num_clusters = 0;
    return coral_common(&cc, pred, xhat_prev, n_tokens, static_cast<char*>(workspace) + L->coral, L->pred - L->coral);
}

// The fp32 prediction from x_hat_l (zero without it) into P: the cross-layer
// kernels with no quantisation stage.  Their error word goes to the fit's.
// The residual's encoding, for the decoder (codes == NULL: none).
struct SasResidual {
    const uint32_t* codes = nullptr;
    const uint32_t* meta = nullptr;
    const uint8_t* ids = nullptr;
    const qvg_bf16* centroids = nullptr;
};

// The layer's prediction (fp32) into P (may be NULL).  Given the residual's
// encoding, the same kernel also forms xhat = bf16(pred + r_hat), r_hat being
// the residual decoded exactly as qvg_decode decodes it.
qvg_status sas_predict(const qvg_config* cfg, const coral_predictor* pred, const qvg_bf16* xhat_prev,
                       int64_t n_tokens, const SasLayout& L, void* workspace, float* P, const SasResidual& r,
                       qvg_bf16* xhat, const FitWorkspace& w, cudaStream_t s) {
    char* base = static_cast<char*>(workspace);
    qvg::CoralArgs a{};
    a.xprev = xhat_prev;
    a.B = xhat_prev ? pred->B : nullptr; a.U = xhat_prev ? pred->U : nullptr; a.W = xhat_prev ? pred->W : nullptr;
    a.R = xhat_prev ? pred->rank : 0;
    a.prepared = xhat_prev ? pred->prepared : nullptr;
    a.n_tokens = n_tokens; a.H = cfg->num_heads;
    a.S = r.codes ? cfg->num_stages : 0;
    a.codes = const_cast<uint32_t*>(r.codes);
    a.meta = const_cast<uint32_t*>(r.meta);
    a.ids = r.ids;
    a.cent = r.centroids;
    a.C = cfg->num_clusters;
    a.xhat = r.codes ? xhat : nullptr;
    a.pred_out = P;
    a.lowrank = reinterpret_cast<float*>(base + L.coral);
    a.workspace = base + L.coral;
    a.workspace_bytes = L.pred - L.coral;
    a.err_out = reinterpret_cast<uint32_t*>(w.stats + 3);
    return cuda_status(qvg::launch_coral(cfg->head_dim, cfg->group_size, false, a, s), "coral prediction launch");
}

qvg_status sas_decode_residual(const qvg_config* cfg, const uint32_t* codes, const uint32_t* meta, const uint8_t* ids,
                               const qvg_bf16* centroids, int64_t n_tokens, qvg_bf16* out, cudaStream_t s) {
    qvg::DecodeArgs d;
    d.codes = codes; d.meta = meta; d.ids = ids; d.cent = centroids;
    d.chunk_offset = nullptr; d.chunk_version = nullptr; d.n_chunks = 0;
    d.cap = n_tokens; d.tok_begin = 0; d.tok_end = n_tokens;
    d.out = out; d.out_head_stride = cfg->head_dim; d.out_token_stride = (int64_t)cfg->num_heads * cfg->head_dim;
    d.H = cfg->num_heads; d.C = cfg->num_clusters; d.S = cfg->num_stages; d.bits = cfg->bits;
    return cuda_status(qvg::launch_decode(cfg->head_dim, cfg->group_size, d, s), "decode launch");
}

}  // namespace

extern "C" {

qvg_status coral_sas_workspace_bytes(const qvg_config* cfg, int64_t n_tokens, size_t* bytes) {
    qvg_status st = check_config(cfg, true);
    if (st) return st;
    if (!bytes || n_tokens < 0) return fail(QVG_ERR_INVALID_ARG, "bad arguments");
    *bytes = sas_layout(cfg, n_tokens).total;
    return ok();
}

qvg_status coral_sas_encode(const qvg_config* cfg, const coral_predictor* pred, const qvg_bf16* xhat_prev,
                            const qvg_bf16* x_next, int64_t n_tokens, uint32_t* codes, uint32_t* meta, uint8_t* ids,
                            qvg_bf16* centroids, qvg_bf16* xhat_next, float* pred_out, void* workspace,
                            size_t workspace_bytes, qvg_stream stream) {
    SasLayout L;
    qvg_status st = sas_check(cfg, pred, xhat_prev, n_tokens, workspace, workspace_bytes, &L);
    if (st) return st;
    if (!x_next || !codes || !meta || !ids || !centroids || !xhat_next) return fail(QVG_ERR_INVALID_ARG, "buffer is NULL");
    if (!aligned16(x_next) || !aligned16(codes) || !aligned16(meta) || !aligned16(centroids) || !aligned16(xhat_next) ||
        !aligned16(pred_out))
        return fail(QVG_ERR_INVALID_ARG, "buffers must be 16-byte aligned");
    cudaStream_t s = (cudaStream_t)stream;
    char* base = static_cast<char*>(workspace);
    FitWorkspace w = carve(cfg, n_tokens, workspace);
    float* P = pred_out ? pred_out : reinterpret_cast<float*>(base + L.pred);
    qvg_bf16* R = reinterpret_cast<qvg_bf16*>(base + L.res);
    const int64_t HD = (int64_t)cfg->num_heads * cfg->head_dim, count = n_tokens * HD;
    cudaError_t e = cudaMemsetAsync(w.stats, 0, sizeof(unsigned long long) * 4, s);
    if (e != cudaSuccess) return cuda_status(e, "memset");
    if ((st = sas_predict(cfg, pred, xhat_prev, n_tokens, L, workspace, P, SasResidual{}, nullptr, w, s))) return st;
    // the residual r = bf16(x_{l+1} - pred), smoothed and quantised like a KV tensor
    if ((e = qvg::launch_coral_residual(x_next, P, count, R, s)) != cudaSuccess) return cuda_status(e, "residual launch");
    e = qvg::launch_kmeans_init(cfg->head_dim, R, cfg->head_dim, HD, n_tokens, nullptr, cfg->num_heads,
                                cfg->num_clusters, centroids, s);
    if (e != cudaSuccess) return cuda_status(e, "init launch");
    if ((st = lloyd(cfg, R, n_tokens, cfg->head_dim, HD, centroids, ids, n_tokens, 0, w, s, false))) return st;
    qvg::EncodeArgs a;
    a.x = R; a.head_stride = cfg->head_dim; a.token_stride = HD; a.n_tokens = n_tokens;
    a.cent = centroids; a.ids = ids;
    a.codes = codes; a.meta = meta; a.cap = n_tokens; a.tok_offset = 0;
    a.H = cfg->num_heads; a.C = cfg->num_clusters; a.S = cfg->num_stages; a.bits = cfg->bits;
    if ((e = qvg::launch_encode(cfg->head_dim, cfg->group_size, a, s)) != cudaSuccess) return cuda_status(e, "encode launch");
    // x_hat_{l+1} = bf16(pred + r_hat), exactly as the decoder forms it
    if ((st = sas_decode_residual(cfg, codes, meta, ids, centroids, n_tokens, R, s))) return st;
    return cuda_status(qvg::launch_coral_recon(P, R, count, xhat_next, s), "reconstruction launch");
}

qvg_status coral_sas_decode(const qvg_config* cfg, const coral_predictor* pred, const qvg_bf16* xhat_prev,
                            int64_t n_tokens, const uint32_t* codes, const uint32_t* meta, const uint8_t* ids,
                            const qvg_bf16* centroids, qvg_bf16* xhat_next, float* pred_out, void* workspace,
                            size_t workspace_bytes, qvg_stream stream) {
    SasLayout L;
    qvg_status st = sas_check(cfg, pred, xhat_prev, n_tokens, workspace, workspace_bytes, &L);
    if (st) return st;
    if (!codes || !meta || !ids || !centroids || !xhat_next) return fail(QVG_ERR_INVALID_ARG, "buffer is NULL");
    if (!aligned16(codes) || !aligned16(meta) || !aligned16(centroids) || !aligned16(xhat_next) || !aligned16(pred_out))
        return fail(QVG_ERR_INVALID_ARG, "buffers must be 16-byte aligned");
    cudaStream_t s = (cudaStream_t)stream;
    FitWorkspace w = carve(cfg, n_tokens, workspace);
    cudaError_t e = cudaMemsetAsync(w.stats, 0, sizeof(unsigned long long) * 4, s);
    if (e != cudaSuccess) return cuda_status(e, "memset");
    // one pass: the prediction kernel decodes the residual (centroid row plus
    // dequantised stages, rounded to bf16) and forms x_hat itself; the fp32
    // prediction is stored only when the caller asks for it
    SasResidual r;
    r.codes = codes; r.meta = meta; r.ids = ids; r.centroids = centroids;
    return sas_predict(cfg, pred, xhat_prev, n_tokens, L, workspace, pred_out, r, xhat_next, w, s);
}

}  // extern "C"

namespace {

// Validates an attention call and fills its arguments; *skip = true when
// there is nothing to launch.
qvg_status attention_args(const qvg_config* cfg, const qvg_bf16* q, int64_t n_queries, int64_t q_head_stride,
                          int64_t q_token_stride, const qvg_encoded_view* k, const qvg_encoded_view* v,
                          int64_t capacity, int64_t n_keys, float scale, float* out, int64_t out_head_stride,
                          int64_t out_token_stride, qvg::AttnArgs* ap, bool* skip) {
    *skip = false;
    qvg_status st = check_config(cfg, false);
    if (st) return st;
    if (cfg->head_dim != 64 && cfg->head_dim != 128)
        return fail(QVG_ERR_UNSUPPORTED, "fused attention supports head_dim 64 or 128 (got %d)", cfg->head_dim);
    if (n_queries < 0) return fail(QVG_ERR_INVALID_ARG, "negative query count");
    if (capacity < 0 || n_keys < 1 || n_keys > capacity)
        return fail(QVG_ERR_INVALID_ARG, "n_keys %lld must be in 1..capacity (%lld)", (long long)n_keys,
                    (long long)capacity);
    if (!std::isfinite(scale)) return fail(QVG_ERR_INVALID_ARG, "scale must be finite");
    if (!k || !v) return fail(QVG_ERR_INVALID_ARG, "k/v encoding is NULL");
    const bool has_c = cfg->num_clusters > 0;
    for (const qvg_encoded_view* e : {k, v}) {
        if (!e->codes || !e->meta) return fail(QVG_ERR_INVALID_ARG, "codes/meta is NULL");
        if (!aligned16(e->codes) || !aligned16(e->meta))
            return fail(QVG_ERR_INVALID_ARG, "codes/meta must be 16-byte aligned");
        if (has_c && (!e->ids || !e->centroids || !aligned16(e->centroids)))
            return fail(QVG_ERR_INVALID_ARG, "ids/centroids missing or centroids not 16-byte aligned");
    }
    if (n_queries == 0) {
        *skip = true;
        return ok();
    }
    if ((st = check_input(cfg, q, n_queries, q_head_stride, q_token_stride, "q"))) return st;
    if (!out || !aligned16(out)) return fail(QVG_ERR_INVALID_ARG, "out must be non-NULL and 16-byte aligned");
    if (out_head_stride % 4 || out_token_stride % 4 || out_head_stride < 0 || out_token_stride < 0)
        return fail(QVG_ERR_INVALID_ARG, "out strides must be non-negative multiples of 4");
    qvg::AttnArgs a;
    a.q = q; a.q_head_stride = q_head_stride; a.q_token_stride = q_token_stride; a.n_queries = n_queries;
    a.k_codes = k->codes; a.k_meta = k->meta; a.k_ids = k->ids; a.k_cent = k->centroids;
    a.v_codes = v->codes; a.v_meta = v->meta; a.v_ids = v->ids; a.v_cent = v->centroids;
    a.cap = capacity; a.n_keys = n_keys;
    a.out = out; a.out_head_stride = out_head_stride; a.out_token_stride = out_token_stride;
    a.H = cfg->num_heads; a.C = cfg->num_clusters; a.S = cfg->num_stages; a.G = cfg->group_size; a.bits = cfg->bits;
    a.scale_log2 = scale * 1.4426950408889634f;
    *ap = a;
    return ok();
}

}  // namespace

extern "C" {

qvg_status qvg_attention_decode(const qvg_config* cfg, const qvg_bf16* q, int64_t n_queries, int64_t q_head_stride,
                                int64_t q_token_stride, const qvg_encoded_view* k, const qvg_encoded_view* v,
                                int64_t capacity, int64_t n_keys, float scale, float* out, int64_t out_head_stride,
                                int64_t out_token_stride, qvg_stream stream) {
    qvg::AttnArgs a;
    bool skip = false;
    qvg_status st = attention_args(cfg, q, n_queries, q_head_stride, q_token_stride, k, v, capacity, n_keys, scale,
                                   out, out_head_stride, out_token_stride, &a, &skip);
    if (st || skip) return st;
    return cuda_status(qvg::launch_attention_decode(cfg->head_dim, a, (cudaStream_t)stream), "attention launch");
}

qvg_status qvg_attention_workspace_bytes(const qvg_config* cfg, int64_t n_keys, size_t* bytes) {
    qvg_status st = check_config(cfg, false);
    if (st) return st;
    if (!bytes) return fail(QVG_ERR_INVALID_ARG, "bytes is NULL");
    if (n_keys < 0) return fail(QVG_ERR_INVALID_ARG, "negative key count");
    *bytes = cfg->head_dim == 128 ? qvg::attention_staged_bytes(cfg->head_dim, cfg->num_heads, n_keys) : 0;
    return ok();
}

qvg_status qvg_attention_decode_staged(const qvg_config* cfg, const qvg_bf16* q, int64_t n_queries,
                                       int64_t q_head_stride, int64_t q_token_stride, const qvg_encoded_view* k,
                                       const qvg_encoded_view* v, int64_t capacity, int64_t n_keys, float scale,
                                       float* out, int64_t out_head_stride, int64_t out_token_stride,
                                       void* workspace, size_t workspace_bytes, qvg_stream stream) {
    qvg::AttnArgs a;
    bool skip = false;
    qvg_status st = attention_args(cfg, q, n_queries, q_head_stride, q_token_stride, k, v, capacity, n_keys, scale,
                                   out, out_head_stride, out_token_stride, &a, &skip);
    if (st || skip) return st;
    const size_t need = cfg->head_dim == 128 ? qvg::attention_staged_bytes(cfg->head_dim, cfg->num_heads, n_keys) : 0;
    if (need && (!workspace || ((uintptr_t)workspace & 255u)))
        return fail(QVG_ERR_INVALID_ARG, "workspace NULL or not 256-byte aligned (need %zu bytes)", need);
    if (workspace_bytes < need) return fail(QVG_ERR_INVALID_ARG, "workspace too small: %zu < %zu bytes", workspace_bytes, need);
    bool launched = false;
    cudaError_t e = qvg::launch_attention_staged(cfg->head_dim, a, workspace, workspace_bytes, &launched, (cudaStream_t)stream);
    if (e == cudaSuccess && !launched) e = qvg::launch_attention_decode(cfg->head_dim, a, (cudaStream_t)stream);
    return cuda_status(e, "attention launch");
}

}  // extern "C"
