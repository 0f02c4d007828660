// attn_f32.cu -- exact attention forward in fp32 on the CUDA cores.
//
// The same online-softmax recurrence as the tensor-core path ("第二十二课…"
// §三十二 pseudo-code; "少搬一趟：FlashAttention 四代进化史" §2.2), kept in fp32 so the
// output meets fp32 accuracy.  Eight threads share one query row: each holds
// d / 8 of its head-dim columns of q and of the unnormalised output
// accumulator in registers; a score is the sum of their eight partial dot
// products (a three-step shuffle tree within the row's lanes), and each of
// them keeps the row's running max m and sum l (the same values in all
// eight) and updates its own columns.  A CTA of 128 threads covers 16
// consecutive query rows of one (sequence, head) and walks the keys in tiles
// of 32 that all its threads read from shared memory.  The key loop stops at
// the last key any row of the CTA can see (causal), and key positions past
// the sequence end are masked ([L22] §三十四–§三十五).
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "../../include/fa.h"
#include "fa_error.cuh"
#include "launch.h"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr int kThreads = 128;
constexpr int kGroup = 8;                    // threads per query row
constexpr int kRows = kThreads / kGroup;     // query rows per CTA
constexpr int kKeys = 32;                    // keys per shared-memory tile
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.69314718055994531f;

struct F32Params {
    const float *Q, *K, *V;
    float *O, *lse;
    int B, H, N, d;
    int64_t total;
    float scale_log2;         // scale * log2(e)
    int causal;
    const int32_t *cu_seqlens;
    int *err_word;
};

// DMAX: compile-time bound on d (32, 64 or 128); d itself may be smaller.
template <int DMAX>
__global__ void __launch_bounds__(kThreads) attn_fwd_f32_kernel(const F32Params p)
{
    constexpr int kCols = DMAX / kGroup;     // head-dim columns per thread
    __shared__ float k_s[kKeys][DMAX];
    __shared__ float v_s[kKeys][DMAX];

    const int qtile = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    int64_t start;
    int L;
    if (p.cu_seqlens) {
        start = p.cu_seqlens[b];
        const int64_t end = p.cu_seqlens[b + 1];
        if (start < 0 || end < start || end > p.total || end - start > p.N) {
            if (threadIdx.x == 0 && qtile == 0 && h == 0)
                record_device_error(p.err_word, FA_DEVERR_BAD_SEQLENS);
            return;
        }
        L = int(end - start);
    } else {
        start = int64_t(b) * p.N;
        L = p.N;
    }
    const int q0 = qtile * kRows;
    if (q0 >= L)
        return;
    const int d = p.d, H = p.H;
    const int r = threadIdx.x / kGroup;      // row in the CTA
    const int g = threadIdx.x % kGroup;      // column group: columns g kCols ..
    const int c0 = g * kCols;
    const int i = q0 + r;                    // query position in the sequence
    const bool row_ok = i < L;

    float q[kCols], acc[kCols];
#pragma unroll
    for (int c = 0; c < kCols; ++c) {
        q[c] = (row_ok && c0 + c < d) ? p.Q[((start + i) * H + h) * d + c0 + c] : 0.f;
        acc[c] = 0.f;
    }
    float m = -INFINITY, l = 0.f;            // m in log2 units of the scaled score

    const int last_q = min(q0 + kRows, L) - 1;
    const int n_keys = p.causal ? last_q + 1 : L;
    // the next tile's K and V are loaded into registers while this one is
    // used, so the loads' latency overlaps the arithmetic
    constexpr int kPer = kKeys * DMAX / kThreads;   // elements per thread and tile
    float kr[kPer], vr[kPer];
    auto load_tile = [&](int j0) {
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
            const int idx = threadIdx.x + u * kThreads;
            const int jj = idx / DMAX, c = idx % DMAX;
            kr[u] = vr[u] = 0.f;
            if (j0 + jj < L && c < d) {
                const int64_t off = ((start + j0 + jj) * H + h) * d + c;
                kr[u] = p.K[off];
                vr[u] = p.V[off];
            }
        }
    };
    load_tile(0);
    for (int j0 = 0; j0 < n_keys; j0 += kKeys) {
        __syncthreads();                     // the previous tile is fully consumed
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
            const int idx = threadIdx.x + u * kThreads;
            k_s[idx / DMAX][idx % DMAX] = kr[u];
            v_s[idx / DMAX][idx % DMAX] = vr[u];
        }
        __syncthreads();
        if (j0 + kKeys < n_keys)
            load_tile(j0 + kKeys);

        float s[kKeys];
        float tmax = -INFINITY;
#pragma unroll
        for (int jj = 0; jj < kKeys; ++jj) {
            float dot = 0.f;
#pragma unroll
            for (int c = 0; c < kCols; ++c)
                dot = fmaf(q[c], k_s[jj][c0 + c], dot);
            // the row's eight partial sums (lanes 8 r' .. 8 r' + 7 of the warp)
            dot += __shfl_xor_sync(0xffffffffu, dot, 1);
            dot += __shfl_xor_sync(0xffffffffu, dot, 2);
            dot += __shfl_xor_sync(0xffffffffu, dot, 4);
            const int j = j0 + jj;
            const bool vis = j < L && (!p.causal || j <= i);
            s[jj] = vis ? dot * p.scale_log2 : -INFINITY;
            tmax = fmaxf(tmax, s[jj]);
        }
        const float m_new = fmaxf(m, tmax);
        if (m_new == -INFINITY)
            continue;                        // nothing visible yet for this row
        const float corr = ptx::ex2(m - m_new);   // 0 on the first visible tile
        l *= corr;
#pragma unroll
        for (int c = 0; c < kCols; ++c)
            acc[c] *= corr;
#pragma unroll
        for (int jj = 0; jj < kKeys; ++jj) {
            const float pj = ptx::ex2(s[jj] - m_new);
            l += pj;
#pragma unroll
            for (int c = 0; c < kCols; ++c)
                acc[c] = fmaf(pj, v_s[jj][c0 + c], acc[c]);
        }
        m = m_new;
    }

    if (!row_ok)
        return;
    const float inv = 1.f / l;
    float *o = p.O + ((start + i) * H + h) * d;
#pragma unroll
    for (int c = 0; c < kCols; ++c)
        if (c0 + c < d)
            o[c0 + c] = acc[c] * inv;
    if (g == 0) {
        const float lse = (m + log2f(l)) * kLn2;
        if (p.cu_seqlens)
            p.lse[int64_t(h) * p.total + start + i] = lse;
        else
            p.lse[(int64_t(b) * H + h) * p.N + i] = lse;
    }
}

}  // namespace

int launch_attention_f32(const AttnArgs &a, cudaStream_t stream)
{
    F32Params p;
    p.Q = static_cast<const float *>(a.Q);
    p.K = static_cast<const float *>(a.K);
    p.V = static_cast<const float *>(a.V);
    p.O = static_cast<float *>(a.O);
    p.lse = a.lse;
    p.B = a.B;
    p.H = a.H;
    p.N = a.N;
    p.d = a.d;
    p.total = a.total;
    p.scale_log2 = float(double(a.scale) * 1.4426950408889634);
    p.causal = a.causal;
    p.cu_seqlens = a.cu_seqlens;
    p.err_word = a.err_word;
    const dim3 grid((a.N + kRows - 1) / kRows, a.H, a.B);
    if (a.d <= 32)
        attn_fwd_f32_kernel<32><<<grid, kThreads, 0, stream>>>(p);
    else if (a.d <= 64)
        attn_fwd_f32_kernel<64><<<grid, kThreads, 0, stream>>>(p);
    else
        attn_fwd_f32_kernel<128><<<grid, kThreads, 0, stream>>>(p);
    return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // namespace fa
