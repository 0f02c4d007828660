// launch.h -- host-side entry points of the kernels, called by fa_api.cu after
// argument validation.  Each returns an FA_* code.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include <mutex>

namespace fa {

// A kernel's dynamic shared-memory limit is raised once per device (the
// attribute belongs to the current device's context): one PerDeviceOnce per
// kernel and call site.
struct PerDeviceOnce {
    static constexpr int kDevices = 64;
    std::once_flag flag[kDevices];
    cudaError_t err[kDevices] = {};
};

inline bool set_max_dynamic_smem(PerDeviceOnce &o, const void *kernel, int bytes)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= PerDeviceOnce::kDevices)
        return false;
    std::call_once(o.flag[dev], [&] {
        o.err[dev] = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          bytes);
    });
    return o.err[dev] == cudaSuccess;
}

// Row softmax of x [rows, N] into y (y may equal x).
int launch_softmax_rows(const float *x, float *y, int64_t rows, int64_t N, cudaStream_t stream);

// Arguments shared by both attention paths.  Layout rules are those of fa.h.
struct AttnArgs {
    const void *Q, *K, *V;
    void *O;
    float *lse;
    int B, H, N, d;
    int H_row = 0;            // heads per token row in memory (0: H); > H for a
                              // view of heads [h0, h0 + H): Q/K/V/O point at head
                              // h0 of row 0, lse at head h0's first entry
    int64_t total;            // packed token count (B * N when dense)
    float scale;
    int causal;
    const int32_t *cu_seqlens;  // device pointer or nullptr (dense)
    int *err_word;            // device error word
    // split-KV (dense bf16 only): keys per sequence, causal offset (query i
    // sees keys j <= i + kv_off), key ranges per Q-tile pair, fp32 scratch
    int Nk = 0;               // 0: same as N
    int kv_off = 0;
    int splits = 1;
    float *O_accum = nullptr; // [splits, B, N, H, d] (packed: [splits, total, H, d])
    float *lse_accum = nullptr;  // [splits, B, H, N] (packed: [splits, H, total])
    // split-KV on packed batches: key rows per sequence; cu_seqlens holds the
    // query rows, total the query row count
    const int32_t *cu_seqlens_k = nullptr;
    int64_t total_k = 0;
    // failure-detection test (fa_debug_expire_next_wait): nonzero makes the
    // bf16 kernel's MMA warp first wait this many ns on a barrier that nothing
    // arrives at, so the wait runs out and every CTA takes its abort path
    uint32_t expire_wait_ns = 0;
};

int launch_attention_bf16(const AttnArgs &a, cudaStream_t stream);
int launch_attention_f32(const AttnArgs &a, cudaStream_t stream);

// Merges `splits` partial results (O_accum, lse_accum as above) into O (bf16,
// [B, N, H, d]) and lse ([B, H, N]).
int launch_attention_combine(const AttnArgs &a, cudaStream_t stream);

// Number of key splits the library picks for a dense problem (>= 1).
int choose_num_splits(int B, int H, int N, int Nk);

// 3-D TMA map over a [total, H, d] bf16 tensor: box = 64 head-dim elements
// (128 bytes, the 128-byte swizzle span) x 1 head x box_rows rows (128 unless
// given); rows past `total` read as zero.  With H_row > 0 the map covers H
// heads of rows that hold H_row heads (a head-range view; base points at its
// first head).  False if the driver refuses the map.
bool make_tmap_bf16(CUtensorMap *tm, const void *base, int64_t total, int H, int d,
                    int box_rows = 128, int H_row = 0);

// TMA maps over the FP8 forward's e4m3 tensors: rows of Q' / K' ([total, H, d]
// bytes, box d x 1 x 128, d = 128 so a row is one 128-byte swizzle span) and
// the transposed V' ([rows = B*H*d, n_pad] bytes, box 128 keys x d rows).
bool make_tmap_e4m3_rows(CUtensorMap *tm, const void *base, int64_t total, int H, int d);
bool make_tmap_e4m3_vt(CUtensorMap *tm, const void *base, int64_t rows, int64_t n_pad, int d);
// 4-D TMA map over a dense [B, N, H, d] tensor (bf16, or e4m3 bytes): box = one
// 128-byte row segment (64 bf16 or 128 e4m3) x 1 head x 128 rows x 1 sequence,
// 128-byte swizzle.  Rows past N of a sequence read as zero and are not stored.
bool make_tmap_seq_4d(CUtensorMap *tm, const void *base, bool e4m3, int B, int N, int H, int d);

// FP8 attention forward on the quantised tensors (dense; d = 128).
struct AttnFp8Args {
    const uint8_t *Qf, *Kf, *Vt;
    const float *sq, *sk, *sv;
    void *O;
    float *lse;
    int B, H, N, d, n_pad;
    float scale;
    int causal;
    int *err_word;
    const int32_t *cu_seqlens = nullptr;  // packed: [B + 1] prefix sums; N = longest
    int64_t total = 0;                    // packed: rows of Q, K, V, O
};
int launch_attention_fp8(const AttnFp8Args &a, cudaStream_t stream);

// Backward of the bf16 attention (dense [B, N, H, d] or packed [total, H, d]);
// layouts as in fa.h.
struct AttnBwdArgs {
    const void *Q, *K, *V, *O, *dO;
    const float *lse;          // [B, H, N] (packed: [H, total]), natural log, from the forward
    void *dQ, *dK, *dV;
    float *D;                  // the same layout as lse, scratch: D_i = dO_i . O_i
    int B, H, N, d;            // packed: N = longest sequence (an upper bound)
    float scale;
    int causal;
    int *err_word;
    const int32_t *cu_seqlens = nullptr;  // packed: device [B + 1] prefix sums
    int64_t total = 0;                    // packed: rows of the tensors
    float *dq_acc = nullptr;              // one-pass form: the workspace (see below)
    // failure-detection test (fa_debug_expire_next_wait), one-pass form only:
    // nonzero makes the tensor-core warp wait that long on a barrier that
    // nothing arrives at, so that the timeout path runs
    uint32_t expire_wait_ns = 0;
};
int launch_attention_bwd(const AttnBwdArgs &a, cudaStream_t stream);
// One-pass backward (d = 64 or 128, dense or packed): dQ summed over the key tiles
// by fp32 atomic adds into the workspace a.dq_acc, then converted.
int launch_attention_bwd_atomic(const AttnBwdArgs &a, cudaStream_t stream);
inline int64_t bwd_atomic_n_pad(int N) { return (int64_t(N) + 63) / 64 * 64; }
// Workspace of the one-pass form (d = 64, 128): the fp32 dQ accumulator [B H,
// n_pad, d], then (lse log2 e, D) pairs [B H, n_pad]; packed batches: the
// accumulator [H, total + 64, d], then the pairs [H, B, n_pad].
inline int64_t bwd_atomic_workspace_bytes(int B, int H, int N, int d)
{
    return int64_t(B) * H * bwd_atomic_n_pad(N) * (d + 2) * 4;
}
inline int64_t bwd_atomic_varlen_workspace_bytes(int B, int H, int N, int64_t total, int d)
{
    return int64_t(H) * (total + 64) * d * 4 + int64_t(H) * B * bwd_atomic_n_pad(N) * 8;
}

// Quantisation pass of the FP8 forward (dense [B, N, H, d] bf16 inputs).
struct Fp8QuantArgs {
    const void *Q, *K, *V;
    const float *signs;        // [d], +-1
    uint8_t *Qf, *Kf;          // [B*N, H, d] e4m3 (Q M, K M over scales)
    uint8_t *Vt;               // [B, H, d, n_pad] e4m3, n_pad = 128 * n_tiles
    float *sq, *sk, *vamax;    // [B, H, n_tiles]
    float *sv;                 // [B, H]
    int B, H, N, d;
    int *err_word;             // device error word (bounded waits)
    const int32_t *cu_seqlens = nullptr;  // packed: [B + 1]; Q, K, V, Qf, Kf [total, H, d]
    int64_t total = 0;
};
int launch_fp8_quantize(const Fp8QuantArgs &a, cudaStream_t stream);

}  // namespace fa
