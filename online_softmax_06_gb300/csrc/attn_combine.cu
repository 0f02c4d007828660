// attn_combine.cu -- merge of split-KV partial results.
//
// When the keys of a Q-tile pair are processed in several splits, split s
// leaves, for every query row, its own normalised output O_s and logsumexp
// lse_s over its keys.  The full result follows from the online-softmax merge
// rule ("第二十二课：Softmax 为什么难以高效…" §十九 and §二十二: m = max(m_A, m_B),
// l = e^{m_A - m} l_A + e^{m_B - m} l_B, and the same weights on the outputs),
// written in logsumexp form:
//     lse = m + ln sum_s exp(lse_s - m),   m = max_s lse_s
//     O   = sum_s exp(lse_s - lse) * O_s
// ("从 FlashAttention 看懂算子融合…": split-KV with per-split outputs and lse,
// then a combine kernel).  One warp per (sequence, query row, head); lanes
// split the splits for the reductions and the head dimension for O.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <type_traits>

#include "../../include/fa.h"
#include "launch.h"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.69314718055994531f;
constexpr int kWarpsPerBlock = 8;

template <int D>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
    attn_combine_kernel(const float *O_accum, const float *lse_accum, __nv_bfloat16 *O,
                        float *lse, int B, int H, int N, int splits)
{
    // Launched as a programmatic dependent of the split kernel: everything
    // above the partials' first read may overlap that kernel's end; the wait
    // returns once the split kernel has completed and its writes are visible.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    constexpr int kPerLane = D / 32;
    const int lane = threadIdx.x & 31;
    const int64_t row = int64_t(blockIdx.x) * kWarpsPerBlock + (threadIdx.x >> 5);
    const int64_t rows = int64_t(B) * N * H;
    if (row >= rows)
        return;
    const int h = int(row % H);
    const int i = int((row / H) % N);
    const int b = int(row / (int64_t(N) * H));
    const int64_t split_stride_lse = int64_t(B) * H * N;
    const int64_t lse_off = (int64_t(b) * H + h) * N + i;

    constexpr int kBatch = 16;
    using Vec = typename std::conditional<kPerLane == 4, float4, float2>::type;
    const int64_t split_stride_o = int64_t(B) * N * H * D;
    const int64_t o_off = row * D + lane * kPerLane;   // row = (b * N + i) * H + h
    // The first kBatch splits' O rows are loaded before the weights are known,
    // so their loads overlap those of the logsumexps.  A split that saw no key
    // of the row (lse_s = -inf) never wrote its O_s: its weight is 0 and its
    // values, whatever they are, are selected away below, never multiplied.
    Vec v0[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u)
        if (u < splits)
            v0[u] = *reinterpret_cast<const Vec *>(O_accum + u * split_stride_o + o_off);

    // m = max_s lse_s; lse = m + ln sum_s exp(lse_s - m)   (log2 units inside).
    // Lane l keeps lse of split l (the first chunk of 32) in a register, so
    // with up to 32 splits every lse is read once.
    const float x0 = lane < splits ? lse_accum[lane * split_stride_lse + lse_off] * kLog2e
                                   : -INFINITY;
    float mx = x0;
    for (int s = lane + 32; s < splits; s += 32)
        mx = fmaxf(mx, lse_accum[s * split_stride_lse + lse_off] * kLog2e);
    for (int o = 16; o > 0; o >>= 1)
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    float sum = 0.f;
    if (mx != -INFINITY) {
        sum = ptx::ex2(x0 - mx);                     // 0 past the last split
        for (int s = lane + 32; s < splits; s += 32)
            sum += ptx::ex2(lse_accum[s * split_stride_lse + lse_off] * kLog2e - mx);
    }
    for (int o = 16; o > 0; o >>= 1)
        sum += __shfl_xor_sync(0xffffffffu, sum, o);
    const float total = (mx == -INFINITY) ? -INFINITY : mx + log2f(sum);   // log2 units

    // O = sum_s w_s O_s with w_s = exp(lse_s - lse).  Lane l holds w of split
    // c0 + l of the current chunk of 32; past the first kBatch splits the
    // splits are taken sixteen at a time with their loads issued before the
    // FMAs, and a split with w = 0 is not read.
    float acc[kPerLane];
#pragma unroll
    for (int e = 0; e < kPerLane; ++e)
        acc[e] = 0.f;
    if (total != -INFINITY) {
        // the early-loaded splits (a selected 0 for those with w = 0, whose
        // values are never multiplied)
        {
            const float w_l = ptx::ex2(x0 - total);   // 0 past the last split
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                const float w = __shfl_sync(0xffffffffu, w_l, u);
                if (u < splits && w != 0.f) {
                    const float *f = reinterpret_cast<const float *>(&v0[u]);
#pragma unroll
                    for (int e = 0; e < kPerLane; ++e)
                        acc[e] = fmaf(w, f[e], acc[e]);
                }
            }
        }
        for (int c0 = 0; c0 < splits; c0 += 32) {
            const int s_l = c0 + lane;
            const float x_l = c0 == 0 ? x0
                                      : (s_l < splits
                                             ? lse_accum[s_l * split_stride_lse + lse_off] * kLog2e
                                             : -INFINITY);
            const float w_l = ptx::ex2(x_l - total);   // 0 past the last split
            const int n = splits - c0 < 32 ? splits - c0 : 32;
            for (int u0 = c0 == 0 ? kBatch : 0; u0 < n; u0 += kBatch) {
                float w[kBatch];
                Vec v[kBatch];
#pragma unroll
                for (int u = 0; u < kBatch; ++u)
                    w[u] = __shfl_sync(0xffffffffu, w_l, (u0 + u) & 31);
#pragma unroll
                for (int u = 0; u < kBatch; ++u) {
                    if (u0 + u >= n)
                        w[u] = 0.f;
                    const Vec *src = reinterpret_cast<const Vec *>(
                        O_accum + (c0 + u0 + u) * split_stride_o + o_off);
                    if (w[u] != 0.f)
                        v[u] = *src;
                    else
                        v[u] = Vec{};
                }
#pragma unroll
                for (int u = 0; u < kBatch; ++u) {
                    const float *f = reinterpret_cast<const float *>(&v[u]);
#pragma unroll
                    for (int e = 0; e < kPerLane; ++e)
                        acc[e] = fmaf(w[u], f[e], acc[e]);
                }
            }
        }
    }
    __nv_bfloat16 *dst = O + o_off;
#pragma unroll
    for (int e = 0; e < kPerLane; e += 2) {
        const uint32_t w = ptx::pack_bf16x2(acc[e], acc[e + 1]);
        *reinterpret_cast<uint32_t *>(dst + e) = w;
    }
    if (lane == 0)
        lse[lse_off] = total * kLn2;
}

}  // namespace

int launch_attention_combine(const AttnArgs &a, cudaStream_t stream)
{
    // a packed batch's partials ([splits, total, H, d], [splits, H, total]) are
    // the dense layout of one sequence of `total` rows
    const bool packed = a.cu_seqlens != nullptr;
    const int B = packed ? 1 : a.B;
    const int64_t N64 = packed ? a.total : a.N;
    if (N64 > 0x7fffffffLL)
        return FA_ERR_TOO_LARGE;
    const int N = int(N64);
    const int64_t rows = int64_t(B) * N * a.H;
    if (rows == 0)
        return FA_OK;
    const int64_t blocks = (rows + kWarpsPerBlock - 1) / kWarpsPerBlock;
    if (blocks > 0x7fffffffLL)
        return FA_ERR_TOO_LARGE;
    auto *O = static_cast<__nv_bfloat16 *>(a.O);
    // programmatic dependent launch: the combine's launch and start overlap
    // the end of the split kernel before it on the stream
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(blocks));
    cfg.blockDim = dim3(kWarpsPerBlock * 32);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e =
        a.d == 64 ? cudaLaunchKernelEx(&cfg, attn_combine_kernel<64>, a.O_accum, a.lse_accum, O,
                                       a.lse, B, a.H, N, a.splits)
                  : cudaLaunchKernelEx(&cfg, attn_combine_kernel<128>, a.O_accum, a.lse_accum, O,
                                       a.lse, B, a.H, N, a.splits);
    return e == cudaSuccess && cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // namespace fa
