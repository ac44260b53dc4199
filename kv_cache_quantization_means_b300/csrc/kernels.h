// Internal launch interface between the C ABI (api.cu) and the kernels.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace qvg {

struct EncodeArgs {
    const uint16_t* x;
    int64_t head_stride, token_stride, n_tokens;
    const uint16_t* cent;   // [H][C][D] or nullptr
    const uint8_t* ids;     // [H][cap], rows tok_offset.. (C > 0)
    uint32_t* codes;        // [S][H][cap][D*bits/32]
    uint32_t* meta;         // [S][H][cap][D/G]
    int64_t cap, tok_offset;
    int H, C, S;
    int bits;               // code width: 2 or 4
};

struct DecodeArgs {
    const uint32_t* codes;
    const uint32_t* meta;
    const uint8_t* ids;
    const uint16_t* cent;         // version 0 table, [V][H][C][D]
    const int64_t* chunk_offset;  // nullptr: single version
    const int32_t* chunk_version;
    int n_chunks;
    int64_t cap, tok_begin, tok_end;
    uint16_t* out;
    int64_t out_head_stride, out_token_stride;
    int H, C, S;
    int bits;                     // code width: 2 or 4
};

struct AssignArgs {
    const uint16_t* x;
    int64_t head_stride, token_stride, n_tokens;
    const uint16_t* cent;   // [H][C][D]
    int C;
    uint8_t* ids;           // [H][cap]
    int64_t cap, tok_offset;
    int* counts;            // [H][C] or nullptr
    unsigned long long* stats;  // [4] refinement counters or nullptr
    uint32_t* err;              // error code of a kernel that gave up a wait, or nullptr
    // ||x_n||^2 per (head, token) [H][n_tokens], fp32 (tensor-core path only):
    // kNormCompute ignores it, kNormStore computes and stores it, kNormLoad
    // reads what an earlier kNormStore call wrote for the same x.
    float* xnorm;
    int xnorm_mode;
    // ids that this assign changes, recorded when chg_parts is not null (the
    // tensor-core path only).  Each CTA records the rows of its token range
    // [start, start + ...) in that range of chg_tok (token) and chg_on (old
    // id | new id << 8), [H][chg_stride] each, and sets chg_parts[h][part] =
    // (start, count); the caller zeroes chg_parts ([H][kChgParts]) first.
    int* chg_tok;
    uint16_t* chg_on;
    int2* chg_parts;
    int64_t chg_stride;     // head stride of chg_tok / chg_on: n_tokens rounded up to a multiple of 8
};
constexpr int kChgParts = 160;   // token ranges (assign CTAs) per head, at most
constexpr int kNormCompute = 0, kNormStore = 1, kNormLoad = 2;

constexpr int kUpdFull = 0, kUpdIncremental = 1;

struct UpdateArgs {
    const uint16_t* x;
    int64_t head_stride, token_stride, n_tokens;
    const uint8_t* ids;     // [H][cap], rows tok_offset..; an id >= C is in no cluster
    int64_t cap, tok_offset;
    int H, C;
    int group_log2;         // clusters per CTA = 2^group_log2 (<= 16), or -1: chosen from H, C and n_tokens
    uint16_t* cent;         // [H][C][D] in/out
    // Exact state that one update leaves for the next: per cluster the
    // fixed-point window sums of its members ([H][C][3][D]) and their count,
    // and per group of clusters a flag that its window sums are not valid (a
    // member value of magnitude >= 2^14).  kUpdFull recomputes and stores
    // all of it; kUpdIncremental applies the changes an assign recorded since
    // the previous update (AssignArgs::chg_*), then rounds the means of the
    // clusters those changes touched.
    long long* ksum;
    int* kcount;
    int* kbig;              // [H][C] (groups of a head use its first entries)
    const int* chg_tok;     // [H][chg_stride]
    const uint16_t* chg_on; // [H][chg_stride]
    const int2* chg_parts;  // [H][kChgParts]
    int64_t chg_stride;
    int mode;
};

struct CoralArgs {
    const uint16_t* xprev;   // [N][H*D] or nullptr
    const uint16_t* xnext;   // [N][H*D] (encode) or nullptr (decode)
    const uint16_t* B;       // [H][D][D]
    const uint16_t* U;       // [H*D][R]
    const uint16_t* W;       // [H*D][R]
    int R;
    int64_t n_tokens;
    int H, S;
    uint32_t* codes;         // [S][H][N][D/16]
    uint32_t* meta;          // [S][H][N][D/G]
    uint16_t* xhat;          // [N][H*D] out, or nullptr: not stored
    float* pred_out;         // optional [N][H*D]
    // decode, optional: the stages code a k-means-smoothed residual (ids [H][N], centroids [H][C][D]);
    // xhat = bf16(pred + bf16(c[id] + stage sum)) instead of bf16(pred + stage sum)
    const uint8_t* ids;
    const uint16_t* cent;
    int C;
    const uint16_t* prepared;  // optional: Wt, then [U | U], as coral_prepare_predictor lays them out
    float* lowrank;          // workspace [N][R]
    void* workspace;         // the whole workspace (tensor-core path)
    size_t workspace_bytes;
    uint32_t* err_out;       // error word of the tensor-core path, or nullptr: the one in its scratch
};

// Scratch of the tensor-core cross-layer path, carved from the workspace.
struct CoralTcScratch {
    uint16_t* t2;      // [N][64] bf16: low-rank projection as (hi, lo) pairs
    uint16_t* wt;      // [32][H*D] bf16: W transposed
    uint16_t* ud;      // [H*D][64] bf16: [U | U]
    uint32_t* err;     // error word (0 = none)
};

// Bytes of CoralTcScratch for H heads of 128 and n_tokens tokens (including
// the error word at the end).
size_t coral_tc_scratch_bytes(int H, int64_t n_tokens);
// The prepared layout of a rank-32 predictor's W and U (H heads of 128):
// Wt [32][H*128], then Ud = [U | U] [H*128][64], each 256-byte aligned.
size_t coral_prepared_bytes(int H);
cudaError_t launch_coral_prep(const uint16_t* W, const uint16_t* U, int H, uint16_t* prepared, cudaStream_t s);
// Points w's Wt and Ud at a prepared layout.
void use_prepared(const uint16_t* prepared, int H, CoralTcScratch& w);

// Each launcher returns cudaSuccess or the launch error; shapes are
// validated by the caller.
cudaError_t launch_encode(int D, int G, const EncodeArgs& a, cudaStream_t s);
cudaError_t launch_decode(int D, int G, const DecodeArgs& a, cudaStream_t s);
// Persistent decoder fed by bulk copies (D = 64 or 128, G >= 16); *launched
// = false (cudaSuccess) when the shape or layout is outside what it handles.
cudaError_t launch_decode_tma(int D, int G, const DecodeArgs& a, bool* launched, cudaStream_t s);
// The device error word of the kernels that take no workspace (read, and
// cleared when `clear`), and the bounded-wait limit / test flags; both
// synchronise `s`.
cudaError_t read_codec_error(uint32_t* out, bool clear, cudaStream_t s);
// That error word's device address on the current device (looked up once per
// device), or nullptr when the lookup fails.
uint32_t* codec_error_word();
cudaError_t set_codec_debug(unsigned long long wait_limit_ns, uint32_t flags, cudaStream_t s);
// What the kernels with bounded waits read at launch: the device error word
// of the current device (0x7E000000 once a wait ran out, for the kernels
// without a workspace), the wait limit in ns and the test flags (bit 0: each
// CTA's copy producer withholds its first copy, so that the first wait on it
// runs out).
struct CodecCtl {
    uint32_t* err;
    unsigned long long limit;
    uint32_t flags;
};
// The current device's control block (the error word's address is looked up
// once per device); false when the lookup fails.
bool codec_ctl(CodecCtl* ctl);
cudaError_t launch_kmeans_init(int D, const uint16_t* x, int64_t head_stride, int64_t token_stride,
                               int64_t n_tokens, const uint16_t* warm, int H, int C, uint16_t* cent,
                               cudaStream_t s);
// *recorded (if not null) says whether the launched kernel records id
// changes (AssignArgs::chg_parts).
cudaError_t launch_assign(int D, int H, const AssignArgs& a, cudaStream_t s, bool* recorded = nullptr);
// tcgen05 assign; sets *launched = false (and returns cudaSuccess) when the
// shape or layout is outside what it handles, so the caller can fall back.
cudaError_t launch_assign_tc(int D, int H, const AssignArgs& a, bool* launched, cudaStream_t s);
cudaError_t launch_update(int D, const UpdateArgs& a, cudaStream_t s);
cudaError_t launch_set_chunk(int64_t* chunk_offset, int32_t* chunk_version, int idx, int64_t begin,
                             int64_t end, int32_t version, cudaStream_t s);
cudaError_t launch_coral(int D, int G, bool encode, const CoralArgs& a, cudaStream_t s);
// Coral + SAS hybrid, element-wise over count (a multiple of 8) elements:
// r = bf16(x_next - pred) and x_hat = bf16(pred + r_hat), fp32 arithmetic.
cudaError_t launch_coral_residual(const uint16_t* xnext, const float* pred, int64_t count, uint16_t* r,
                                  cudaStream_t s);
cudaError_t launch_coral_recon(const float* pred, const uint16_t* rhat, int64_t count, uint16_t* xhat,
                               cudaStream_t s);
// tcgen05 cross-layer path (D = 128, rank 32, G <= 64, a previous layer);
// *launched = false (cudaSuccess) when outside that set.
cudaError_t launch_coral_tc(int D, int G, bool encode, const CoralArgs& a, const CoralTcScratch& w, bool* launched,
                            cudaStream_t s);

// The low-rank stage alone (W^T / [U|U] layout and t = x_hat W as bf16
// hi/lo pairs into w.t2); D = 128, R = 32, 128-byte aligned scratch.
cudaError_t launch_coral_lowrank_tc(const CoralArgs& a, const CoralTcScratch& w, cudaStream_t s);

// Adapted block predictors: per head the ridge least-squares block of
// y - U t = B x_hat (D = 128, R = 32), from x_hat, y = x_{l+1} and t2
// (launch_coral_lowrank_tc).  part: coral_fit_part_bytes scratch.
constexpr int kFitChunkTokens = 1024;   // tokens per fp32 partial Gram sum
size_t coral_fit_part_bytes(int H, int64_t n_tokens);
cudaError_t launch_coral_fit(const uint16_t* xh, const uint16_t* y, const uint16_t* t2, const uint16_t* U,
                             int64_t n_tokens, int H, float* part, uint16_t* B, cudaStream_t s);

}  // namespace qvg
