/*
 * qvg.h -- C ABI of the B300 KV-cache codec (libqvg.so).
 *
 * Two codecs for the key/value cache of an autoregressive video diffusion
 * model, after the pages they come from:
 *
 *  - Quant VideoGen (QVG; gist.science explainer of arXiv 2602.02958,
 *    "Sommario tecnico"): semantic-aware smoothing (sec. 2A: per-head k-means
 *    along the sequence axis, subtraction of each token's centroid) followed
 *    by progressive residual quantisation (sec. 2B: several stages of 2-bit
 *    quantisation, each coding what the previous stages left; decoding
 *    dequantises, sums the stages and adds the centroid back).  Centroid
 *    caching (sec. 3) gives the streaming append call.
 *  - Coral-KV (news items on the preprint, section "cross-layer
 *    prediction"): layer l+1 is predicted from the reconstruction of layer l
 *    by a block-diagonal-per-head plus global low-rank (block-DPLR) map and
 *    only the prediction residual is quantised.
 *
 * Conventions for every call
 *  - Pointers named x, centroids, codes, meta, ids, out, workspace, B, U, W,
 *    xhat_* and pred are DEVICE pointers into caller-owned memory; the library
 *    never allocates, frees or synchronises.  A qvg_config / qvg_cache /
 *    coral_predictor struct itself lives in host memory.
 *  - bf16 and fp16 values travel as their 16-bit patterns (qvg_bf16).
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *    stream) and returns before it runs.  Calls are capturable in a CUDA graph
 *    except qvg_append_chunk, whose host-side bookkeeping happens at call time.
 *  - Arguments are validated on the host before anything is launched; a bad
 *    argument returns QVG_ERR_INVALID_ARG (or QVG_ERR_UNSUPPORTED for a shape
 *    outside the supported set, QVG_ERR_CAPACITY for a full cache) and
 *    launches nothing.  A failed launch returns QVG_ERR_CUDA.  The message of
 *    the last failure on the calling thread is qvg_last_error().  No C++
 *    exception crosses this boundary.
 *
 * Supported shapes: head_dim D in {32, 64, 128, 256} (k-means: D <= 128);
 * group_size G in {16, 32, 64, 128} dividing D; num_stages S in 1..4;
 * bits b = 2 (the QVG codec) or 4 (the PRQ_INT4 variant named by the KV
 * Cache Quantization for Self-Forcing Video Generation study, read as the same
 * group scheme with 15 steps; the cross-layer codec is 2-bit only);
 * num_clusters C in 0..256 (0 = no smoothing).  Pointers must be 16-byte
 * aligned and strides multiples of 8 elements.
 *
 * Encoded layout of one (layer, tensor) with `capacity` token rows per head:
 *   codes : uint32 [S][H][capacity][D*b/32]; element j of a row sits in word
 *           j/(32/b), bits b*(j%(32/b)) .. b*(j%(32/b))+b-1 (least
 *           significant first).
 *   meta  : uint32 [S][H][capacity][D/G]; low half = fp16 scale s =
 *           fp16((max - min) / (2^b - 1)), high half = fp16 zero-point z of
 *           the group; a code q decodes to q*s + z.
 *   ids   : uint8  [H][capacity] cluster of each token row (C > 0 only).
 *   centroids : bf16 [V][H][C][D], V centroid-table versions (V = 1 unless
 *           streaming).
 * Compressed bits per element = S*b + 32*S/G + [C > 0]*(8/D + 16*C*V/N).
 */
#ifndef QVG_H
#define QVG_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define QVG_API __attribute__((visibility("default")))
#else
#define QVG_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t qvg_bf16;
typedef void* qvg_stream;

typedef enum {
    QVG_OK = 0,
    QVG_ERR_INVALID_ARG = 1,
    QVG_ERR_UNSUPPORTED = 2,
    QVG_ERR_CAPACITY = 3,
    QVG_ERR_CUDA = 4,
    QVG_ERR_TIMEOUT = 5
} qvg_status;

typedef struct {
    int32_t num_heads;     /* H */
    int32_t head_dim;      /* D */
    int32_t num_clusters;  /* C, 0 = no smoothing */
    int32_t lloyd_iters;   /* T, Lloyd iterations of qvg_fit_centroids */
    int32_t num_stages;    /* S */
    int32_t bits;          /* bits per code: 2 or 4 (cross-layer codec: 2) */
    int32_t group_size;    /* G, elements per (scale, zero) along D */
} qvg_config;

/* Streaming cache of one (layer, tensor).  Device buffers are caller-owned;
 * the counters are host-side state that qvg_append_chunk advances. */
typedef struct {
    uint32_t* codes;         /* [S][H][capacity][D/16] */
    uint32_t* meta;          /* [S][H][capacity][D/G]  */
    uint8_t* ids;            /* [H][capacity]          */
    qvg_bf16* centroids;     /* [max_versions][H][C][D] */
    int64_t* chunk_offset;   /* device [max_chunks + 1], first token of chunk i; [n_chunks] = n_used */
    int32_t* chunk_version;  /* device [max_chunks], centroid version of chunk i */
    int64_t capacity;        /* token rows per head */
    int32_t max_versions;
    int32_t max_chunks;      /* <= 4096 */
    int64_t n_used;          /* tokens appended so far (host) */
    int32_t n_versions;      /* centroid tables written so far (host) */
    int32_t n_chunks;        /* chunks appended so far (host) */
} qvg_cache;

/* Block-DPLR predictor of layer l+1 from layer l (Coral-KV):
 * pred[n][h*D+o] = sum_i B[h][o][i] x[n][h*D+i] + sum_r U[h*D+o][r] t[n][r],
 * t[n][r] = sum_j W[j][r] x[n][j].  All bf16, device. */
typedef struct {
    const qvg_bf16* B;   /* [H][D][D] (out x in) */
    const qvg_bf16* U;   /* [H*D][R] */
    const qvg_bf16* W;   /* [H*D][R] */
    int32_t rank;        /* R, 0 = block-diagonal only; R % 16 == 0, R <= 64 */
    /* Optional (NULL: none): U and W already laid out for the tensor-core
     * path by coral_prepare_predictor, so that no call re-lays them out.  It
     * depends on U and W only, so it stays valid when B is refit. */
    const qvg_bf16* prepared;
} coral_predictor;

/* Message of the last failed call on this thread ("" if none). */
QVG_API const char* qvg_last_error(void);

/* Library version string. */
QVG_API const char* qvg_version(void);

/* Bytes of each encoded buffer for `capacity` token rows and `n_versions`
 * centroid tables (host only; any output pointer may be NULL).  Follows the
 * layout above; ids and centroids are 0 when C = 0. */
QVG_API qvg_status qvg_encoded_bytes(const qvg_config* cfg, int64_t capacity, int32_t n_versions,
                             size_t* codes_bytes, size_t* meta_bytes, size_t* ids_bytes,
                             size_t* centroid_bytes);

/* Scratch bytes that qvg_fit_centroids / qvg_encode / qvg_update /
 * qvg_append_chunk / coral_* need for `n_tokens` tokens (host only). */
QVG_API qvg_status qvg_workspace_bytes(const qvg_config* cfg, int64_t n_tokens, size_t* bytes);

/* Diagnostics of the last k-means call (fit, assign, update, append) that
 * used `workspace`: out[0] = token rows the tensor-core screen could not
 * decide and re-ranked exactly, out[1] = those among them whose nearest
 * centroid was settled by exact squared distances, out[2] = those among
 * them that needed the channel-order fp64 sum (near-exact ties),
 * out[3] = error word (0 = none; 0x7E000000 = a kernel gave up waiting on an
 * internal barrier and its ids are not valid).  With C = 0 (a Coral-KV
 * configuration) out[0..2] are 0 and out[3] is the error word of the last
 * coral_* call that used `workspace` (0x7E000000 = a tensor-core kernel gave
 * up waiting and its outputs are not valid).  Returns QVG_ERR_TIMEOUT (with
 * out filled) when the error word is set, QVG_OK otherwise.  Copies from the
 * device and waits for `stream`; out is host memory. */
QVG_API qvg_status qvg_fit_stats(const qvg_config* cfg, int64_t n_tokens, const void* workspace,
                         size_t workspace_bytes, uint64_t* out, qvg_stream stream);

/* Error word of the kernels that take no workspace -- the persistent PRQ
 * decoder behind qvg_decode, qvg_decode_cache and coral_sas_*, and the
 * tensor-core kernels of coral_predict_encode_static: 0 = none,
 * 0x7E000000 = a kernel gave up one of its bounded waits (about 2 s by
 * default) and the outputs of that call are not valid.  The word is shared by every call on the current device and keeps
 * its value until cleared; clear != 0 resets it to 0 after reading.  Returns
 * QVG_ERR_TIMEOUT (with *out filled) when the word was set, QVG_OK when it
 * was 0.  Waits for `stream`; out is host memory. */
QVG_API qvg_status qvg_device_error(uint32_t* out, int32_t clear, qvg_stream stream);

/* Test hook of the bounded waits of the kernels above and of the
 * tensor-core k-means assign: wait_limit_ns is the limit after which a
 * waiting role gives up (0 restores the default, 2 s); flags bit 0 makes each
 * CTA's copy producer withhold its first copy, so that the first wait of that
 * CTA's consumers runs out (and the call records 0x7E000000 -- in the device
 * error word, or for the assign in the workspace word that qvg_fit_stats
 * reads -- drains its other copies and returns).  For failure-path tests
 * only; waits for `stream`, then applies to every call the process makes
 * afterwards. */
QVG_API qvg_status qvg_debug_set_wait(uint64_t wait_limit_ns, uint32_t flags, qvg_stream stream);

/* SAS k-means (QVG sec. 2A items 1-2 and sec. 3): per head, T Lloyd iterations
 * of (assign, update) on the n_tokens rows of x.  x is bf16 with logical
 * layout [H][n_tokens][D]: row (h, n) starts at x + h*head_stride +
 * n*token_stride (elements; D contiguous).  Initial centroids are
 * warm_start ([H][C][D]) when non-NULL, else the tokens floor(j*n/C).
 * Writes the last update's centroids ([H][C][D]) and the last assignment's
 * ids to ids[h*capacity + tok_offset + n].  Assignment is the exact argmin of
 * the squared Euclidean distance (lowest index on ties); an empty cluster
 * keeps its centroid; a centroid is the exact mean of its tokens rounded to
 * bf16.  Needs n_tokens >= 1 and C >= 1.  `workspace` (qvg_workspace_bytes)
 * must not be shared with concurrent calls. */
QVG_API qvg_status qvg_fit_centroids(const qvg_config* cfg, const qvg_bf16* x, int64_t n_tokens,
                             int64_t head_stride, int64_t token_stride, const qvg_bf16* warm_start,
                             qvg_bf16* centroids, uint8_t* ids, int64_t capacity, int64_t tok_offset,
                             void* workspace, size_t workspace_bytes, qvg_stream stream);

/* Assign step alone: ids[h*capacity + tok_offset + n] = argmin_j ||x - c_j||^2. */
QVG_API qvg_status qvg_assign(const qvg_config* cfg, const qvg_bf16* x, int64_t n_tokens,
                      int64_t head_stride, int64_t token_stride, const qvg_bf16* centroids,
                      uint8_t* ids, int64_t capacity, int64_t tok_offset, void* workspace,
                      size_t workspace_bytes, qvg_stream stream);

/* Update step alone: centroids (in/out, [H][C][D]) <- mean of their tokens
 * under ids; empty clusters unchanged. */
QVG_API qvg_status qvg_update(const qvg_config* cfg, const qvg_bf16* x, int64_t n_tokens,
                      int64_t head_stride, int64_t token_stride, const uint8_t* ids,
                      int64_t capacity, int64_t tok_offset, qvg_bf16* centroids, void* workspace,
                      size_t workspace_bytes, qvg_stream stream);

/* QVG encode (sec. 2A item 3 and sec. 2B items 1-2): per token row,
 * r = x - c[id] in fp32 (r = x when C = 0), then for each stage and group of G
 * channels s = fp16((max r - min r)/3), z = fp16(min r),
 * q = clamp(rint((r - z) / s), 0, 3) with IEEE single-precision division (0 when
 * s = 0), r <- r - (q*s + z).
 * Rows go to rows tok_offset .. tok_offset+n_tokens-1 of codes/meta/ids.
 * assign = 0: ids are read from `ids` (e.g. written by qvg_fit_centroids);
 * assign = 1: ids are first computed against `centroids` and written there. */
QVG_API qvg_status qvg_encode(const qvg_config* cfg, const qvg_bf16* x, int64_t n_tokens,
                      int64_t head_stride, int64_t token_stride, const qvg_bf16* centroids,
                      int32_t assign, uint32_t* codes, uint32_t* meta, uint8_t* ids,
                      int64_t capacity, int64_t tok_offset, void* workspace, size_t workspace_bytes,
                      qvg_stream stream);

/* QVG decode (sec. 2B item 3): rows [tok_begin, tok_end) of every head,
 * x_hat = bf16(((c[id] + d_1) + d_2) + ...), d_s = q_s*s_s + z_s in fp32,
 * written to out + h*out_head_stride + (n - tok_begin)*out_token_stride. */
QVG_API qvg_status qvg_decode(const qvg_config* cfg, const uint32_t* codes, const uint32_t* meta,
                      const uint8_t* ids, const qvg_bf16* centroids, int64_t capacity,
                      int64_t tok_begin, int64_t tok_end, qvg_bf16* out, int64_t out_head_stride,
                      int64_t out_token_stride, qvg_stream stream);

/* Streaming append (centroid caching, QVG sec. 3): encodes n_new new tokens
 * at row cache->n_used.  refit != 0: the chunk is fitted (T iterations,
 * warm-started from the newest table, cold when there is none) and the result
 * is pushed as a new table version; refit == 0: the chunk's tokens are
 * assigned to the newest table.  Advances n_used, n_chunks (and n_versions).
 * QVG_ERR_CAPACITY if rows, chunks or versions would overflow. */
QVG_API qvg_status qvg_append_chunk(const qvg_config* cfg, qvg_cache* cache, const qvg_bf16* x,
                            int64_t n_new, int64_t head_stride, int64_t token_stride,
                            int32_t refit, void* workspace, size_t workspace_bytes,
                            qvg_stream stream);

/* Decode rows [tok_begin, tok_end) of a streaming cache, each chunk against
 * its own centroid version. */
QVG_API qvg_status qvg_decode_cache(const qvg_config* cfg, const qvg_cache* cache, int64_t tok_begin,
                            int64_t tok_end, qvg_bf16* out, int64_t out_head_stride,
                            int64_t out_token_stride, qvg_stream stream);

/* Coral-KV closed-loop encode of one layer (cfg->num_clusters must be 0):
 * pred = block-DPLR(xhat_prev) in fp32 (0 when xhat_prev is NULL: first
 * layer), r = x_next - pred, PRQ-coded per head row into codes/meta
 * ([S][H][n_tokens][...]), and xhat_next = bf16(((pred + d_1) + d_2) + ...)
 * written for the next layer.  xhat_prev, x_next, xhat_next are token-major
 * [n_tokens][H*D].  pred_out ([n_tokens][H*D] fp32) may be NULL; when given it
 * receives the prediction (for staged checks). */
QVG_API qvg_status coral_predict_encode(const qvg_config* cfg, const coral_predictor* pred,
                                const qvg_bf16* xhat_prev, const qvg_bf16* x_next, int64_t n_tokens,
                                uint32_t* codes, uint32_t* meta, qvg_bf16* xhat_next, float* pred_out,
                                void* workspace, size_t workspace_bytes, qvg_stream stream);

/* Allocation-free variant of coral_predict_encode.  The paper has no
 * counterpart to this call: it is an interface convenience for callers that
 * cannot allocate device memory or pass a workspace -- a runtime whose
 * allocator owns all device memory, a plugin that must not grow the
 * footprint, or code that cannot call cudaMalloc at the point of use.  Arguments and results are those
 * of coral_predict_encode without the workspace: the low-rank scratch is a
 * fixed 4 MiB device array inside this library (64 floats per token), which
 * every GPU that loads the library keeps until the process exits.
 *  - n_tokens must be <= 16384, and the call's scratch (the low-rank
 *    projection or, with head_dim 128 and rank 32, the tensor-core path's
 *    128*n_tokens + 192*H*D bytes and a little alignment, whichever is
 *    larger) must fit the 4 MiB; otherwise QVG_ERR_CAPACITY, launching
 *    nothing.  The call allocates and frees nothing.
 *  - The first call on a device (with a previous layer) looks up the array's
 *    device address, and that of the library's device error word, on the
 *    current device; make that first call before any stream capture.
 *  - All calls share the one array: calls whose work can overlap on the GPU
 *    (other streams, other host threads) race and must be serialised by the
 *    caller.  The array's contents carry nothing from one call to the next:
 *    each call writes every value it reads before reading it.
 *  - A tensor-core wait that runs out (its outputs are then not valid) is
 *    recorded in the library's device error word: read it with
 *    qvg_device_error. */
QVG_API qvg_status coral_predict_encode_static(const qvg_config* cfg, const coral_predictor* pred,
                                       const qvg_bf16* xhat_prev, const qvg_bf16* x_next, int64_t n_tokens,
                                       uint32_t* codes, uint32_t* meta, qvg_bf16* xhat_next, float* pred_out,
                                       qvg_stream stream);

/* Adapted configuration of the cross-layer codec (Coral-KV pages: the light
 * block-diagonal predictors are rebuilt for the current video, the low-rank
 * part stays as calibrated).  Per head h, the ridge least-squares block
 *   B_h = argmin_B sum_n ||y_{n,h} - U_h t_n - B xhat_{n,h}||^2 + lambda_h ||B||^2,
 *   t_n = W^T xhat_n, lambda_h = 2^-20 trace(X_h^T X_h) / D,
 * from xhat_prev (= xhat_l, bf16 [n_tokens][H*D]) and x_next (= x_{l+1}, same
 * layout), written to B_out (bf16 [H][D][D], B[h][o][i]; device memory,
 * caller-owned).  pred supplies U and W (rank 32; pred->B is not read).  The
 * block is then used as the predictor's B for coral_predict_encode of this
 * layer, and must be stored with the stream so that the decoder uses the same
 * one.  Sums: bf16 products, fp32 accumulation per 1024-token chunk, chunks
 * added in a fixed order, fp32 Cholesky solve; B_h = 0 when X_h is zero.
 * Needs C = 0, D = 128, rank 32, n_tokens >= 1 and qvg_workspace_bytes of
 * workspace (256-byte aligned); qvg_fit_stats reports its error word. */
/* Bytes of the prepared layout of a rank-32 predictor's U and W for H heads
 * of D = 128 (W transposed, then [U | U], each 256-byte aligned). */
QVG_API qvg_status coral_prepared_bytes(const qvg_config* cfg, int32_t rank, size_t* bytes);

/* Writes that layout of pred->U and pred->W (rank 32, head_dim 128) into
 * `prepared` (device, caller-owned, 256-byte aligned, coral_prepared_bytes
 * long).  Setting pred->prepared to it afterwards lets every call skip the
 * re-layout (bit-identical results).  Errors: invalid arguments return an
 * error code and launch nothing; asynchronous on `stream`. */
QVG_API qvg_status coral_prepare_predictor(const qvg_config* cfg, const coral_predictor* pred, qvg_bf16* prepared,
                                           size_t prepared_bytes, qvg_stream stream);

QVG_API qvg_status coral_fit_block(const qvg_config* cfg, const coral_predictor* pred, const qvg_bf16* xhat_prev,
                                   const qvg_bf16* x_next, int64_t n_tokens, qvg_bf16* B_out, void* workspace,
                                   size_t workspace_bytes, qvg_stream stream);

/* Decoder twin of coral_predict_encode: rebuilds xhat_next from xhat_prev,
 * the predictor and the stored codes (bit-identical to the encoder's
 * xhat_next). */
QVG_API qvg_status coral_predict_decode(const qvg_config* cfg, const coral_predictor* pred,
                                const qvg_bf16* xhat_prev, int64_t n_tokens, const uint32_t* codes,
                                const uint32_t* meta, qvg_bf16* xhat_next, float* pred_out,
                                void* workspace, size_t workspace_bytes, qvg_stream stream);

/* Coral-KV + SAS hybrid: the cross-layer prediction (Coral-KV pages, the
 * block-diagonal plus low-rank predictor of layer l+1 from the reconstructed
 * layer l) combined with the k-means smoothing of Quant VideoGen (Sommario
 * tecnico sec. 2A), applied to the prediction residual.  The pages do not
 * describe the combination; this library's reading, per layer:
 *   pred  = block-DPLR(xhat_prev) in fp32 (0 when xhat_prev is NULL),
 *   r     = bf16(x_next - pred)            (fp32 difference, then RN to bf16),
 *   centroids, ids = k-means of r per head (init + T Lloyd steps, as
 *                    qvg_fit_centroids), codes/meta = PRQ of r - c[id]
 *                    (as qvg_encode),
 *   r_hat = the decoded residual (as qvg_decode), xhat_next = bf16(pred + r_hat).
 * cfg: num_clusters C >= 1, lloyd_iters >= 1, bits 2, head_dim 64 or 128.
 * Buffers (device memory, caller-owned, 16-byte aligned): xhat_prev, x_next,
 * xhat_next token-major bf16 [n_tokens][H*D]; codes [S][H][n_tokens][D/16],
 * meta [S][H][n_tokens][D/G], ids [H][n_tokens], centroids bf16 [H][C][D];
 * pred_out fp32 [n_tokens][H*D] or NULL (receives the prediction).
 * workspace: coral_sas_workspace_bytes of it, 256-byte aligned; it begins
 * with the k-means workspace, so qvg_fit_stats(cfg, n_tokens, workspace, ...)
 * reports the re-rank counters and the error word of both the k-means and the
 * cross-layer kernels.  Errors: invalid arguments return an error code and
 * launch nothing; asynchronous. */
QVG_API qvg_status coral_sas_workspace_bytes(const qvg_config* cfg, int64_t n_tokens, size_t* bytes);

QVG_API qvg_status coral_sas_encode(const qvg_config* cfg, const coral_predictor* pred, const qvg_bf16* xhat_prev,
                                    const qvg_bf16* x_next, int64_t n_tokens, uint32_t* codes, uint32_t* meta,
                                    uint8_t* ids, qvg_bf16* centroids, qvg_bf16* xhat_next, float* pred_out,
                                    void* workspace, size_t workspace_bytes, qvg_stream stream);

/* Decoder twin of coral_sas_encode: xhat_next = bf16(pred + r_hat) from
 * xhat_prev, the predictor and the stored codes, meta, ids and centroids
 * (bit-identical to the encoder's xhat_next).  One pass: the prediction
 * kernel decodes r_hat itself (centroid row plus dequantised stages, rounded
 * to bf16 as qvg_decode rounds it) and adds it to the prediction, so no
 * residual buffer is written and the fp32 prediction only when pred_out is
 * non-NULL. */
QVG_API qvg_status coral_sas_decode(const qvg_config* cfg, const coral_predictor* pred, const qvg_bf16* xhat_prev,
                                    int64_t n_tokens, const uint32_t* codes, const uint32_t* meta, const uint8_t* ids,
                                    const qvg_bf16* centroids, qvg_bf16* xhat_next, float* pred_out,
                                    void* workspace, size_t workspace_bytes, qvg_stream stream);

/* One encoded (layer, tensor) as qvg_encode writes it (single centroid
 * version); device pointers, caller-owned. */
typedef struct {
    const uint32_t* codes;       /* [S][H][capacity][D*b/32] */
    const uint32_t* meta;        /* [S][H][capacity][D/G] */
    const uint8_t* ids;          /* [H][capacity]; NULL when C == 0 */
    const qvg_bf16* centroids;   /* [H][C][D]; NULL when C == 0 */
} qvg_encoded_view;

/* Attention over a compressed K/V history with the decode fused in (Quant
 * VideoGen explainer, sec. 3: fused dequantisation kernels; the 33-method
 * Self-Forcing KV-cache study, abstract: rebuilt BF16 K/V buffers around
 * attention undo the memory saving).  No bf16 K or V buffer is written.
 * For every head h and query i < n_queries (non-causal: every query sees
 * keys 0 .. n_keys-1 of the head):
 *   s_n = scale * <q_i, k_hat_n>,
 *   out_i = sum_n exp(s_n) v_hat_n / sum_n exp(s_n),
 * where k_hat and v_hat are, bit for bit, the bf16 rows that qvg_decode
 * writes for rows 0 .. n_keys-1 of the encodings k and v (both with cfg's
 * S, b, G, C).  Arithmetic: bf16 products of q and k_hat with fp32 sums,
 * fp32 online softmax, probabilities rounded to bf16 for the product with
 * v_hat, fp32 sums; out is fp32.
 * q: bf16 at q + h*q_head_stride + i*q_token_stride (strides multiples of 8
 * elements, 16-byte aligned).  out: fp32 at out + h*out_head_stride +
 * i*out_token_stride (strides multiples of 4 elements, 16-byte aligned).
 * Needs head_dim 64 or 128 (QVG_ERR_UNSUPPORTED otherwise), 1 <= n_keys <=
 * capacity, a finite scale.  n_queries == 0 launches nothing.  Errors:
 * invalid arguments return an error code and launch nothing; asynchronous. */
QVG_API qvg_status qvg_attention_decode(const qvg_config* cfg, const qvg_bf16* q, int64_t n_queries,
                                        int64_t q_head_stride, int64_t q_token_stride, const qvg_encoded_view* k,
                                        const qvg_encoded_view* v, int64_t capacity, int64_t n_keys, float scale,
                                        float* out, int64_t out_head_stride, int64_t out_token_stride,
                                        qvg_stream stream);

/* One (layer, tensor) end to end from host memory, all on `stream`: the copy
 * of x from host to device (x_host holds the layout x_dev will have: the
 * (n_tokens-1)*token_stride + (H-1)*head_stride + D elements from its start,
 * ideally pinned), qvg_fit_centroids (C > 0; warm_start may be NULL), then
 * qvg_encode with those ids, then (out_dev not NULL) qvg_decode of all rows
 * into out_dev with x's strides, and the copy of the encoding to host_out:
 * codes, meta, ids, centroids back to back, each sized as qvg_encoded_bytes
 * gives for capacity = n_tokens and one version.  codes, meta, ids and
 * centroids are device buffers of that size; the workspace is the fit's.
 * Asynchronous: host_out is complete, and x_host free, when the stream
 * reaches this point. */
QVG_API qvg_status qvg_compress_host(const qvg_config* cfg, const qvg_bf16* x_host, qvg_bf16* x_dev, int64_t n_tokens,
                                     int64_t head_stride, int64_t token_stride, const qvg_bf16* warm_start,
                                     qvg_bf16* centroids, uint8_t* ids, uint32_t* codes, uint32_t* meta,
                                     qvg_bf16* out_dev, void* host_out, size_t host_out_bytes, void* workspace,
                                     size_t workspace_bytes, qvg_stream stream);

/* Bytes of the working buffer of qvg_attention_decode_staged for n_keys keys/* Bytes of the working buffer of qvg_attention_decode_staged for n_keys keys
 * (0 when the tensor-core path does not apply: head_dim != 128).  Host only. */
QVG_API qvg_status qvg_attention_workspace_bytes(const qvg_config* cfg, int64_t n_keys, size_t* bytes);

/* The attention of qvg_attention_decode, same arguments and result
 * definition, on the tensor cores (tcgen05) for head_dim 128: each group of
 * up to four heads is first decoded into the caller's working buffer (K as
 * rows, V transposed: 2 * min(H, 4) * n_keys * 128 bf16, sized by
 * qvg_attention_workspace_bytes, 256-byte aligned) -- one decode of every key
 * row per head, with a buffer small enough to stay in L2 rather than a bf16
 * K/V of the whole history -- then 128-query tiles attend to it: S = QK^T and
 * O += PV accumulate in tensor memory, the online softmax in fp32 runs one
 * query row per thread, and its probabilities are rounded to bf16 for the
 * product with v_hat.  The running maximum is raised only when a tile's
 * exceeds it by more than a factor 2^8 (O is then rescaled); the stale
 * maximum scales numerator and denominator alike.  Other head dims, and
 * layouts the bulk copies cannot express, run qvg_attention_decode's kernel.
 * A bounded wait that runs out records 0x7E000000 in the device error word
 * (qvg_device_error).  Asynchronous; the buffer is reused group after group
 * in stream order. */
QVG_API qvg_status qvg_attention_decode_staged(const qvg_config* cfg, const qvg_bf16* q, int64_t n_queries,
                                               int64_t q_head_stride, int64_t q_token_stride,
                                               const qvg_encoded_view* k, const qvg_encoded_view* v,
                                               int64_t capacity, int64_t n_keys, float scale, float* out,
                                               int64_t out_head_stride, int64_t out_token_stride, void* workspace,
                                               size_t workspace_bytes, qvg_stream stream);

#ifdef __cplusplus
}
#endif

#endif /* QVG_H */
