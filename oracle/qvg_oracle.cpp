// QVG / Coral-KV reference oracle -- TEST INFRASTRUCTURE ONLY.
//
// A plain, slow, single-threaded CPU statement of what the KV-cache codec
// computes.  Only the tests, the smoke check and the bench's CPU-baseline leg
// may load it; the product path never does.  It shares no code, header or
// table with the CUDA library.  Compile with -O2 -ffp-contract=off (no
// fast-math) so that every float/double operation below is one IEEE operation
// in the order written.
//
// Sources (web pages; section names as they appear there):
//  * "Quant VideoGen: Auto-Regressive Long Video Generation via 2-Bit
//    KV-Cache Quantization" (gist.science explainer), Sommario tecnico
//    sec. 2A "Semantic-Aware Smoothing" items 1-3 (k-means along the sequence
//    axis, per-group mean, subtraction), sec. 2B "Progressive Residual
//    Quantization" items 1-3 (re-quantise what is left, stage by stage;
//    decoding dequantises and adds the centroids back), sec. 3 (centroid
//    caching), title (2-bit).
//  * "Coral-KV ..." news items (ru / pt), section "cross-layer prediction":
//    layer l predicts layer l+1 through a block-diagonal-per-head plus global
//    low-rank (block-DPLR) map; only the prediction residual is quantised.
//    Section "where cluster quantisation breaks": later frames read the
//    compressed history, which gives the closed-loop reading (predict from
//    the reconstruction).
//
// Readings where the pages are silent (all stated here and in the design
// notes): squared-Euclidean distance; init c_j = x[floor(j*N/C)]; an
// iteration is assign then update, ids from the last assign, centroids from
// the last update; argmin ties go to the lowest index; an empty cluster keeps
// its centroid; centroids are bf16; asymmetric 2-bit group quantiser with an
// fp16 scale s = fp16((max-min)/3) and an fp16 float zero-point z = fp16(min),
// q = clamp(rint((r - z) / s), 0, 3) with IEEE single-precision division
// (q = 0 when s = 0), stage
// residual r <- r - (q*s + z); decoding sums ((c + d1) + d2) + ... in fp32 and
// rounds once to bf16; 16 codes per 32-bit word, least significant first.
//
// Parity pins for every function live in tests/test_oracle_pins.py.

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

namespace {

// ---------------------------------------------------------------- formats --

double bf16_value(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    std::memcpy(&f, &u, 4);
    return (double)f;
}

float bf16_float(uint16_t b) { return (float)bf16_value(b); }

// Round a finite double to the nearest value of a binary format with
// `mant_bits` stored significand bits and minimum normal exponent `min_exp`
// (ties to even), by scaling to the quantum of the value's binade.
double round_to_format(double a, int mant_bits, int min_exp) {
    if (a == 0.0) return a;
    double mag = std::fabs(a);
    int e;
    std::frexp(mag, &e);          // mag = m * 2^e, m in [0.5, 1)
    int binade = e - 1;           // mag in [2^binade, 2^(binade+1))
    if (binade < min_exp) binade = min_exp;
    double quantum = std::ldexp(1.0, binade - mant_bits);
    double n = mag / quantum;     // exact (power-of-two scaling)
    double r = std::nearbyint(n); // default rounding mode: ties to even
    double v = r * quantum;       // exact
    return a < 0 ? -v : v;
}

uint16_t f32_bits_to_bf16(float f) {
    uint32_t u;
    std::memcpy(&u, &f, 4);
    return (uint16_t)(u >> 16);
}

// fp32/fp64 -> bf16, round to nearest even (finite inputs).
uint16_t to_bf16(double a) {
    double v = round_to_format(a, 7, -126);
    if (std::fabs(v) > 3.3895313892515355e38) v = a < 0 ? -INFINITY : INFINITY;
    return f32_bits_to_bf16((float)v);   // v is a bf16 value: exact in fp32
}

// fp32 -> fp16, round to nearest even.
uint16_t to_f16(float f) {
    double a = (double)f;
    uint16_t sign = std::signbit(a) ? 0x8000 : 0;
    double mag = std::fabs(a);
    if (mag >= 65520.0) return sign | 0x7C00;            // rounds to infinity
    double v = round_to_format(mag, 10, -14);
    if (v == 0.0) return sign;
    int e;
    std::frexp(v, &e);
    int binade = e - 1;
    if (binade < -14)                                      // subnormal
        return sign | (uint16_t)(v / std::ldexp(1.0, -24));
    uint16_t mant = (uint16_t)(v / std::ldexp(1.0, binade - 10)) - 1024;
    return sign | (uint16_t)((binade + 15) << 10) | mant;
}

float f16_float(uint16_t h) {
    int sign = (h >> 15) & 1, ex = (h >> 10) & 31, man = h & 1023;
    double v;
    if (ex == 0) v = std::ldexp((double)man, -24);
    else if (ex == 31) v = man ? NAN : INFINITY;
    else v = std::ldexp(1024.0 + man, ex - 25);
    return (float)(sign ? -v : v);
}

// ------------------------------------------------------- SAS: k-means ------

// Squared Euclidean distance in fp64, channels in order 0..D-1.
double sq_dist(const uint16_t* x, const uint16_t* c, int D) {
    double acc = 0.0;
    for (int i = 0; i < D; ++i) {
        double diff = bf16_value(x[i]) - bf16_value(c[i]);
        double sq = diff * diff;
        acc = acc + sq;
    }
    return acc;
}

}  // namespace

extern "C" {

// Format helpers exported so that the tests can pin them.
uint16_t or_to_bf16(double a) { return to_bf16(a); }
uint16_t or_to_f16(float f) { return to_f16(f); }
float or_f16_to_f32(uint16_t h) { return f16_float(h); }

// k-means initialisation: c_j = x[floor(j*N/C)]  (reading of "init from
// tokens at stride N/C").
void or_kmeans_init(const uint16_t* x, int64_t N, int D, int C, uint16_t* cent) {
    for (int j = 0; j < C; ++j) {
        int64_t n = ((int64_t)j * N) / C;
        std::memcpy(cent + (int64_t)j * D, x + n * D, sizeof(uint16_t) * D);
    }
}

// Assign step (SAS item 1): id_n = argmin_j ||x_n - c_j||^2, lowest j on ties.
void or_assign(const uint16_t* x, int64_t N, int D, const uint16_t* cent, int C,
               int32_t* ids, double* dmin) {
    for (int64_t n = 0; n < N; ++n) {
        double best = INFINITY;
        int32_t arg = 0;
        for (int j = 0; j < C; ++j) {
            double d = sq_dist(x + n * D, cent + (int64_t)j * D, D);
            if (d < best) { best = d; arg = j; }
        }
        ids[n] = arg;
        if (dmin) dmin[n] = best;
    }
}

// Update step (SAS item 2): c_j = mean of the tokens assigned to j, summed in
// fp64 in token order, divided in fp64, rounded to bf16.  Empty clusters keep
// their centroid.
void or_update(const uint16_t* x, int64_t N, int D, const int32_t* ids, int C,
               uint16_t* cent, int64_t* counts_out) {
    std::vector<double> sum((size_t)C * D, 0.0);
    std::vector<int64_t> cnt(C, 0);
    for (int64_t n = 0; n < N; ++n) {
        int j = ids[n];
        cnt[j] += 1;
        for (int i = 0; i < D; ++i)
            sum[(size_t)j * D + i] = sum[(size_t)j * D + i] + bf16_value(x[n * D + i]);
    }
    for (int j = 0; j < C; ++j) {
        if (counts_out) counts_out[j] = cnt[j];
        if (cnt[j] == 0) continue;
        for (int i = 0; i < D; ++i)
            cent[(size_t)j * D + i] = to_bf16(sum[(size_t)j * D + i] / (double)cnt[j]);
    }
}

// Lloyd loop: T x (assign, update).  warm == nullptr -> init from tokens.
// Output ids are those of the last assign; centroids those of the last update.
void or_fit(const uint16_t* x, int64_t N, int D, int C, int T, const uint16_t* warm,
            uint16_t* cent, int32_t* ids) {
    if (warm) std::memcpy(cent, warm, sizeof(uint16_t) * (size_t)C * D);
    else or_kmeans_init(x, N, D, C, cent);
    for (int t = 0; t < T; ++t) {
        or_assign(x, N, D, cent, C, ids, nullptr);
        or_update(x, N, D, ids, C, cent, nullptr);
    }
}

// ---------------------------------------------------- PRQ: the encoder -----

// One stage of b-bit asymmetric group quantisation of the fp32 residual r
// (length D, groups of G), in place: r <- r - deq.  L = 2^b - 1 levels above
// the zero-point: s = fp16(range / L), q = clamp(rint((r - z) / s), 0, L).
// b = 2 is the QVG codec (sec. 2B); b = 4 is the Study's PRQ_INT4 variant,
// read as the same scheme with 15 steps.  Writes D*b/32 code words (element e
// at bits b*e of the row, least significant first) and D/G meta words (low
// half = fp16 scale, high half = fp16 zero-point).
static void quantize_stage(float* r, int D, int G, int b, uint32_t* codes, uint32_t* meta) {
    const int L = (1 << b) - 1;
    for (int w = 0; w < D * b / 32; ++w) codes[w] = 0;
    for (int g = 0; g < D / G; ++g) {
        float mn = r[g * G], mx = r[g * G];
        for (int j = 1; j < G; ++j) {
            float v = r[g * G + j];
            if (v < mn) mn = v;
            if (v > mx) mx = v;
        }
        // a zero extreme is taken as +0 (the sign of a zero minimum would
        // otherwise depend on which equal element was seen first)
        mn = mn + 0.0f;
        mx = mx + 0.0f;
        float range = mx - mn;
        float s32 = range / (float)L;
        uint16_t sh = to_f16(s32), zh = to_f16(mn);
        float s = f16_float(sh), z = f16_float(zh);
        meta[g] = (uint32_t)sh | ((uint32_t)zh << 16);
        for (int j = 0; j < G; ++j) {
            int e = g * G + j;
            float t = (s != 0.0f) ? (r[e] - z) / s : 0.0f;
            float qf = std::nearbyint(t);
            int q = qf > 0.0f ? (qf > (float)L ? L : (int)qf) : 0;   // NaN -> 0
            float deq = (float)q * s + z;          // q*s is exact: one rounding
            r[e] = r[e] - deq;
            codes[(e * b) / 32] |= (uint32_t)q << ((e * b) % 32);
        }
    }
}

// QVG encode of one head: r0 = x - c[id] (fp32), then S stages of b-bit
// codes (PRQ items 1-2).  cent/ids may be null (no smoothing, C = 0).
// codes: [S][N][D*b/32]; meta: [S][N][D/G].
void or_prq_encode(const uint16_t* x, int64_t N, int D, const uint16_t* cent,
                   const int32_t* ids, int S, int G, int b, uint32_t* codes, uint32_t* meta) {
    const int W = D * b / 32;
    std::vector<float> r(D);
    for (int64_t n = 0; n < N; ++n) {
        for (int i = 0; i < D; ++i) {
            float xv = bf16_float(x[n * D + i]);
            float cv = cent ? bf16_float(cent[(int64_t)ids[n] * D + i]) : 0.0f;
            r[i] = xv - cv;
        }
        for (int s = 0; s < S; ++s)
            quantize_stage(r.data(), D, G, b, codes + ((int64_t)s * N + n) * W,
                           meta + ((int64_t)s * N + n) * (D / G));
    }
}

// Dequantised contribution of one stage for element e of a row (b-bit codes).
static float stage_value(const uint32_t* codes, const uint32_t* meta, int e, int G, int b) {
    uint32_t q = (codes[(e * b) / 32] >> ((e * b) % 32)) & ((1u << b) - 1u);
    uint32_t m = meta[e / G];
    float s = f16_float((uint16_t)(m & 0xFFFF));
    float z = f16_float((uint16_t)(m >> 16));
    return (float)q * s + z;
}

// QVG decode of one head (PRQ item 3): x_hat = bf16(((c + d1) + d2) + ...).
void or_decode(const uint32_t* codes, const uint32_t* meta, const int32_t* ids,
               const uint16_t* cent, int64_t N, int D, int S, int G, int b, uint16_t* out) {
    const int W = D * b / 32;
    for (int64_t n = 0; n < N; ++n) {
        for (int i = 0; i < D; ++i) {
            float acc = cent ? bf16_float(cent[(int64_t)ids[n] * D + i]) : 0.0f;
            for (int s = 0; s < S; ++s)
                acc = acc + stage_value(codes + ((int64_t)s * N + n) * W,
                                        meta + ((int64_t)s * N + n) * (D / G), i, G, b);
            out[n * D + i] = to_bf16((double)acc);
        }
    }
}

// Streaming rollout of one head (centroid caching, sec. 3): chunk t covers
// tokens [t*chunk, (t+1)*chunk).  When t % refit_every == 0 the chunk is fitted
// (T iterations, warm-started from the latest table, cold at t = 0) and a new
// table version is pushed; otherwise its tokens are assigned to the latest
// table.  Then the chunk is encoded against its version.
// versions: [steps][C][D] (only the first n_versions used); chunk_version:
// [steps]; codes [S][steps*chunk][D*b/32], meta [S][steps*chunk][D/G].
int or_stream(const uint16_t* x, int64_t chunk, int steps, int refit_every, int D, int C,
              int T, int S, int G, int b, uint16_t* versions, int32_t* chunk_version,
              int32_t* ids, uint32_t* codes, uint32_t* meta) {
    int64_t Ntot = chunk * steps;
    const int W = D * b / 32;
    int nv = 0;
    std::vector<uint32_t> cbuf((size_t)S * chunk * W), mbuf((size_t)S * chunk * (D / G));
    for (int t = 0; t < steps; ++t) {
        const uint16_t* xc = x + (int64_t)t * chunk * D;
        int32_t* idc = ids + (int64_t)t * chunk;
        if (t % refit_every == 0) {
            const uint16_t* warm = nv ? versions + (size_t)(nv - 1) * C * D : nullptr;
            or_fit(xc, chunk, D, C, T, warm, versions + (size_t)nv * C * D, idc);
            nv += 1;
        } else {
            or_assign(xc, chunk, D, versions + (size_t)(nv - 1) * C * D, C, idc, nullptr);
        }
        chunk_version[t] = nv - 1;
        or_prq_encode(xc, chunk, D, versions + (size_t)(nv - 1) * C * D, idc, S, G, b,
                      cbuf.data(), mbuf.data());
        for (int s = 0; s < S; ++s) {
            std::memcpy(codes + ((int64_t)s * Ntot + (int64_t)t * chunk) * W,
                        cbuf.data() + (size_t)s * chunk * W, sizeof(uint32_t) * chunk * W);
            std::memcpy(meta + ((int64_t)s * Ntot + (int64_t)t * chunk) * (D / G),
                        mbuf.data() + (size_t)s * chunk * (D / G), sizeof(uint32_t) * chunk * (D / G));
        }
    }
    return nv;
}

// ------------------------------------------------ Coral-KV: block-DPLR -----

// pred[n][h*D+o] = sum_i B[h][o][i] xh[n][h*D+i] + sum_r U[h*D+o][r] t[n][r],
// t[n][r] = sum_j W[j][r] xh[n][j]; fp64, sums in index order.
// xh: [N][H*D] bf16; B: [H][D][D]; U, W: [H*D][R].
void or_coral_predict(const uint16_t* xh, int64_t N, int H, int D, const uint16_t* B,
                      const uint16_t* U, const uint16_t* W, int R, double* pred) {
    int HD = H * D;
    std::vector<double> t(R);
    for (int64_t n = 0; n < N; ++n) {
        const uint16_t* xr = xh + n * HD;
        for (int r = 0; r < R; ++r) {
            double acc = 0.0;
            for (int j = 0; j < HD; ++j) acc = acc + bf16_value(W[(int64_t)j * R + r]) * bf16_value(xr[j]);
            t[r] = acc;
        }
        for (int h = 0; h < H; ++h) {
            for (int o = 0; o < D; ++o) {
                double blk = 0.0;
                for (int i = 0; i < D; ++i)
                    blk = blk + bf16_value(B[((int64_t)h * D + o) * D + i]) * bf16_value(xr[h * D + i]);
                double low = 0.0;
                for (int r = 0; r < R; ++r) low = low + bf16_value(U[((int64_t)h * D + o) * R + r]) * t[r];
                pred[n * HD + h * D + o] = blk + low;
            }
        }
    }
}

// One closed-loop layer of the cross-layer codec.  The prediction (fp64, held
// as fp32 -- or the caller's fp32 prediction `pred_in` when given, for staged
// checks) is subtracted from the true next layer, the residual is PRQ-coded
// per head row (no smoothing), and the reconstruction
// x_hat_next = bf16(((pred + d1) + d2) + ...) is written for the next layer.
// xh_prev == nullptr: layer 0, prediction 0.
// codes: [S][H][N][D/16]; meta: [S][H][N][D/G]; x_next/xh_next: [N][H*D].
void or_coral_encode_layer(const uint16_t* xh_prev, const uint16_t* x_next, int64_t N, int H,
                           int D, const uint16_t* B, const uint16_t* U, const uint16_t* W, int R,
                           const float* pred_in, int S, int G, uint32_t* codes, uint32_t* meta,
                           uint16_t* xh_next, float* pred_out) {
    int HD = H * D;
    std::vector<double> pred64;
    if (xh_prev && !pred_in) {
        pred64.resize((size_t)N * HD);
        or_coral_predict(xh_prev, N, H, D, B, U, W, R, pred64.data());
    }
    std::vector<float> r(D), p(D);
    std::vector<uint32_t> cw((size_t)S * (D / 16)), mw((size_t)S * (D / G));
    for (int64_t n = 0; n < N; ++n) {
        for (int h = 0; h < H; ++h) {
            for (int i = 0; i < D; ++i) {
                int64_t e = n * HD + h * D + i;
                float pv = 0.0f;
                if (pred_in) pv = pred_in[e];
                else if (xh_prev) pv = (float)pred64[e];
                p[i] = pv;
                if (pred_out) pred_out[e] = pv;
                r[i] = bf16_float(x_next[e]) - pv;
            }
            for (int s = 0; s < S; ++s)
                quantize_stage(r.data(), D, G, 2, cw.data() + (size_t)s * (D / 16), mw.data() + (size_t)s * (D / G));
            for (int s = 0; s < S; ++s) {
                std::memcpy(codes + (((int64_t)s * H + h) * N + n) * (D / 16), cw.data() + (size_t)s * (D / 16),
                            sizeof(uint32_t) * (D / 16));
                std::memcpy(meta + (((int64_t)s * H + h) * N + n) * (D / G), mw.data() + (size_t)s * (D / G),
                            sizeof(uint32_t) * (D / G));
            }
            for (int i = 0; i < D; ++i) {
                float acc = p[i];
                for (int s = 0; s < S; ++s) acc = acc + stage_value(cw.data() + (size_t)s * (D / 16),
                                                                    mw.data() + (size_t)s * (D / G), i, G, 2);
                xh_next[n * HD + h * D + i] = to_bf16((double)acc);
            }
        }
    }
}

// Decoder twin of or_coral_encode_layer: rebuilds x_hat_next from x_hat_prev,
// the predictor and the stored codes.
void or_coral_decode_layer(const uint16_t* xh_prev, int64_t N, int H, int D, const uint16_t* B,
                           const uint16_t* U, const uint16_t* W, int R, const float* pred_in, int S,
                           int G, const uint32_t* codes, const uint32_t* meta, uint16_t* xh_next) {
    int HD = H * D;
    std::vector<double> pred64;
    if (xh_prev && !pred_in) {
        pred64.resize((size_t)N * HD);
        or_coral_predict(xh_prev, N, H, D, B, U, W, R, pred64.data());
    }
    for (int64_t n = 0; n < N; ++n)
        for (int h = 0; h < H; ++h)
            for (int i = 0; i < D; ++i) {
                int64_t e = n * HD + h * D + i;
                float acc = pred_in ? pred_in[e] : (xh_prev ? (float)pred64[e] : 0.0f);
                for (int s = 0; s < S; ++s)
                    acc = acc + stage_value(codes + (((int64_t)s * H + h) * N + n) * (D / 16),
                                            meta + (((int64_t)s * H + h) * N + n) * (D / G), i, G, 2);
                xh_next[e] = to_bf16((double)acc);
            }
}

// -------------------------------- Coral-KV: adapted block predictors -----

// Adapted configuration of the Coral-KV pages: the per-head block B_h of the
// predictor is rebuilt for the current video while the offline low-rank part
// (U, W) is kept.  Reading: per head h, B_h minimises
//     sum_n || y_{n,h} - L_{n,h} - B x_{n,h} ||^2 + lambda_h ||B||_F^2,
// with x = the reconstruction x_hat_l, y = x_{l+1}, L = U_h t_n the low-rank
// part of the prediction (t_n = W^T x_hat_n) and a tiny ridge
// lambda_h = 2^-20 * trace(G_h) / D that only matters for (near-)singular
// G_h = X_h^T X_h.  Normal equations: (G_h + lambda_h I) Z = X_h^T (Y_h - L_h)
// with Z = B_h^T, solved by Cholesky; B_h = 0 when X_h is all zero.  Every
// sum is fp64 in token order; the result is rounded to bf16 (the predictor's
// format).  z_out (optional, fp64 [H][D][D], Z before rounding) serves the
// pins.  B_out: bf16 [H][D][D], B[h][o][i].
void or_coral_fit_block(const uint16_t* xh, const uint16_t* y, int64_t N, int H, int D, const uint16_t* U,
                        const uint16_t* W, int R, uint16_t* B_out, double* z_out) {
    const int HD = H * D;
    std::vector<double> t((size_t)N * (R > 0 ? R : 1), 0.0);
    for (int64_t n = 0; n < N; ++n)
        for (int r = 0; r < R; ++r) {
            double acc = 0.0;
            for (int j = 0; j < HD; ++j) acc = acc + bf16_value(W[(int64_t)j * R + r]) * bf16_value(xh[n * HD + j]);
            t[(size_t)n * R + r] = acc;
        }
    std::vector<double> Gm((size_t)D * D), rhs((size_t)D * D), res(D);
    for (int h = 0; h < H; ++h) {
        std::fill(Gm.begin(), Gm.end(), 0.0);
        std::fill(rhs.begin(), rhs.end(), 0.0);
        for (int64_t n = 0; n < N; ++n) {
            const uint16_t* xr = xh + n * HD + h * D;
            // residual target y - L of this token
            for (int o = 0; o < D; ++o) {
                double low = 0.0;
                for (int r = 0; r < R; ++r) low = low + bf16_value(U[((int64_t)h * D + o) * R + r]) * t[(size_t)n * R + r];
                res[o] = bf16_value(y[n * HD + h * D + o]) - low;
            }
            for (int i = 0; i < D; ++i) {
                const double xi = bf16_value(xr[i]);
                for (int k = 0; k < D; ++k) Gm[(size_t)i * D + k] = Gm[(size_t)i * D + k] + xi * bf16_value(xr[k]);
                for (int o = 0; o < D; ++o) rhs[(size_t)i * D + o] = rhs[(size_t)i * D + o] + xi * res[o];
            }
        }
        double tr = 0.0;
        for (int i = 0; i < D; ++i) tr = tr + Gm[(size_t)i * D + i];
        uint16_t* Bh = B_out + (size_t)h * D * D;
        if (tr == 0.0) {
            for (int k = 0; k < D * D; ++k) Bh[k] = 0;
            if (z_out) for (int k = 0; k < D * D; ++k) z_out[(size_t)h * D * D + k] = 0.0;
            continue;
        }
        const double lambda = std::ldexp(tr / D, -20);
        for (int i = 0; i < D; ++i) Gm[(size_t)i * D + i] = Gm[(size_t)i * D + i] + lambda;
        // Cholesky: G = L L^T, L lower triangular, stored in place
        for (int j = 0; j < D; ++j) {
            double d = Gm[(size_t)j * D + j];
            for (int k = 0; k < j; ++k) d = d - Gm[(size_t)j * D + k] * Gm[(size_t)j * D + k];
            d = std::sqrt(d);
            Gm[(size_t)j * D + j] = d;
            for (int i = j + 1; i < D; ++i) {
                double v = Gm[(size_t)i * D + j];
                for (int k = 0; k < j; ++k) v = v - Gm[(size_t)i * D + k] * Gm[(size_t)j * D + k];
                Gm[(size_t)i * D + j] = v / d;
            }
        }
        // for each output channel o: L u = rhs[:, o], then L^T z = u
        for (int o = 0; o < D; ++o) {
            for (int i = 0; i < D; ++i) {
                double v = rhs[(size_t)i * D + o];
                for (int k = 0; k < i; ++k) v = v - Gm[(size_t)i * D + k] * res[k];
                res[i] = v / Gm[(size_t)i * D + i];
            }
            for (int i = D - 1; i >= 0; --i) {
                double v = res[i];
                for (int k = i + 1; k < D; ++k) v = v - Gm[(size_t)k * D + i] * rhs[(size_t)k * D + o];
                rhs[(size_t)i * D + o] = v / Gm[(size_t)i * D + i];   // column o now holds z
            }
        }
        for (int o = 0; o < D; ++o)
            for (int i = 0; i < D; ++i) {
                const double z = rhs[(size_t)i * D + o];                // Z[i][o] = B[o][i]
                Bh[(size_t)o * D + i] = to_bf16(z);
                if (z_out) z_out[((size_t)h * D + o) * D + i] = z;
            }
    }
}

// ------------------------------------------------------------- sizes -------

// Closed-form compressed size in bits per element of one (layer, tensor):
// codes S*b, meta 32*S/G (fp16 scale + fp16 zero per group and stage),
// ids 8/D per element when C > 0 (one byte per token row), centroids
// 16*C*V/N (V table versions of C rows of D bf16 per head, over N tokens).
double or_bits_per_element(int S, int b, int G, int C, int D, int64_t N, int V) {
    double bits = (double)S * b + 32.0 * S / G;
    if (C > 0) bits += 8.0 / D + 16.0 * C * V / (double)N;
    return bits;
}

}  // extern "C"
