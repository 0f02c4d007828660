// softmax.cu -- numerically stable row softmax, y = exp(x - max) / sum exp(x - max).
//
// The kernels follow the stable-softmax lesson ("第二十二课：Softmax 为什么难以高效…",
// lincklin.cn): shift by the row maximum (§二), one max reduction and one sum
// reduction (§三), one warp or one block per row depending on the length
// (§五–§九), and two-level warp-shuffle / shared-memory reductions (§十), with the
// row kept in registers so every element is read from and written to HBM once
// (§十一).  GB300 specifics: 128-bit loads and stores, xor-butterfly shuffles
// (every lane ends with the result, no broadcast step), exp via ex2 on the
// special-function unit, and for long rows a thread-block cluster that splits
// one row across several CTAs and reduces through distributed shared memory,
// so more rows are in flight per SM.  Rows too long for the on-chip budget
// take a two-pass path that reads the row twice and merges per-thread
// (max, sum) pairs with the online-softmax rule (§十九).
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "../../include/fa.h"
#include "launch.h"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float warp_max(float v, int width)
{
    for (int o = width / 2; o > 0; o >>= 1)
        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ float warp_sum(float v, int width)
{
    for (int o = width / 2; o > 0; o >>= 1)
        v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Distributed shared memory: read a float from the same smem variable of CTA
// `rank` of this cluster.
__device__ __forceinline__ float dsmem_load(const float *local, uint32_t rank)
{
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
                 : "=r"(remote)
                 : "r"(ptx::smem_u32(local)), "r"(rank));
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
    return v;
}

__device__ __forceinline__ void cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t cluster_rank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Row softmax with the row resident in registers.
//   G   threads that share one row part: G <= 32 is a sub-warp group (CTA/G rows
//       per CTA, shuffle-only reductions); G == CTA is the whole block (warp
//       shuffles, then shared memory across warps).
//   V   slots per thread; a slot is 4 consecutive floats (one 128-bit access when
//       VEC, four scalar accesses otherwise).  A part covers P = G*V*4 elements
//       and thread t owns slots at element offsets (v*G + t)*4, so each slot
//       index is one fully coalesced pass over the part.
//   CL  CTAs per row (a thread-block cluster; 1 = no cluster).  Only with G == CTA.
template <int G, int V, int CTA, int CL, bool VEC>
__global__ void __launch_bounds__(CTA) softmax_rows_kernel(const float *x, float *y,
                                                           int64_t rows, int64_t N)
{
    static_assert(G <= 32 || G == CTA, "group is a sub-warp or the whole block");
    static_assert(CL == 1 || G == CTA, "clusters split whole-block rows only");
    constexpr int P = G * V * 4;
    constexpr int kWarps = CTA / 32;

    __shared__ float red_max[kWarps];
    __shared__ float red_sum[kWarps];
    __shared__ float cl_max, cl_sum, bc_max, bc_sum;

    int64_t row;
    int t, part;
    if (G <= 32) {
        row = int64_t(blockIdx.x) * (CTA / G) + threadIdx.x / G;
        t = threadIdx.x % G;
        part = 0;
    } else {
        row = int64_t(blockIdx.x) / CL;
        t = threadIdx.x;
        part = (CL > 1) ? int(cluster_rank()) : 0;
    }
    // Rows past the end still take part in the shuffles; they load nothing.
    const bool row_ok = row < rows;
    const int64_t base = row_ok ? row * N : 0;
    const int64_t part0 = int64_t(part) * P;

    float4 v[V];
    float mx = -INFINITY;
#pragma unroll
    for (int s = 0; s < V; ++s) {
        const int64_t e = part0 + int64_t(s * G + t) * 4;
        if (VEC) {
            if (row_ok && e < N)
                v[s] = *reinterpret_cast<const float4 *>(x + base + e);
            else
                v[s] = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
        } else {
            v[s].x = (row_ok && e + 0 < N) ? x[base + e + 0] : -INFINITY;
            v[s].y = (row_ok && e + 1 < N) ? x[base + e + 1] : -INFINITY;
            v[s].z = (row_ok && e + 2 < N) ? x[base + e + 2] : -INFINITY;
            v[s].w = (row_ok && e + 3 < N) ? x[base + e + 3] : -INFINITY;
        }
        mx = fmaxf(mx, fmaxf(fmaxf(v[s].x, v[s].y), fmaxf(v[s].z, v[s].w)));
    }

    // ---- row maximum --------------------------------------------------------
    if (G <= 32) {
        mx = warp_max(mx, G);
    } else {
        mx = warp_max(mx, 32);
        if ((threadIdx.x & 31) == 0)
            red_max[threadIdx.x >> 5] = mx;
        __syncthreads();
        mx = red_max[0];
#pragma unroll
        for (int w = 1; w < kWarps; ++w)
            mx = fmaxf(mx, red_max[w]);
        if (CL > 1) {
            if (threadIdx.x == 0)
                cl_max = mx;
            cluster_sync();
            if (threadIdx.x < 32) {
                float m2 = threadIdx.x < CL ? dsmem_load(&cl_max, threadIdx.x) : -INFINITY;
                m2 = warp_max(m2, 32);
                if (threadIdx.x == 0)
                    bc_max = m2;
            }
            __syncthreads();
            mx = bc_max;
        }
    }

    // ---- exp and row sum (in registers) -------------------------------------
    const float mshift = mx * kLog2e;
    float sum = 0.f;
#pragma unroll
    for (int s = 0; s < V; ++s) {
        v[s].x = ptx::ex2(fmaf(v[s].x, kLog2e, -mshift));
        v[s].y = ptx::ex2(fmaf(v[s].y, kLog2e, -mshift));
        v[s].z = ptx::ex2(fmaf(v[s].z, kLog2e, -mshift));
        v[s].w = ptx::ex2(fmaf(v[s].w, kLog2e, -mshift));
        sum += (v[s].x + v[s].y) + (v[s].z + v[s].w);
    }
    if (G <= 32) {
        sum = warp_sum(sum, G);
    } else {
        sum = warp_sum(sum, 32);
        if ((threadIdx.x & 31) == 0)
            red_sum[threadIdx.x >> 5] = sum;
        __syncthreads();
        float s2 = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w)
            s2 += red_sum[w];
        sum = s2;
        if (CL > 1) {
            if (threadIdx.x == 0)
                cl_sum = sum;
            cluster_sync();
            if (threadIdx.x < 32) {
                float t2 = threadIdx.x < CL ? dsmem_load(&cl_sum, threadIdx.x) : 0.f;
                t2 = warp_sum(t2, 32);
                if (threadIdx.x == 0)
                    bc_sum = t2;
            }
            __syncthreads();
            sum = bc_sum;
        }
    }

    // ---- normalise and store ------------------------------------------------
    const float inv = __frcp_rn(sum);
#pragma unroll
    for (int s = 0; s < V; ++s) {
        const int64_t e = part0 + int64_t(s * G + t) * 4;
        float4 o = make_float4(v[s].x * inv, v[s].y * inv, v[s].z * inv, v[s].w * inv);
        if (VEC) {
            if (row_ok && e < N)
                *reinterpret_cast<float4 *>(y + base + e) = o;
        } else {
            if (row_ok && e + 0 < N) y[base + e + 0] = o.x;
            if (row_ok && e + 1 < N) y[base + e + 1] = o.y;
            if (row_ok && e + 2 < N) y[base + e + 2] = o.z;
            if (row_ok && e + 3 < N) y[base + e + 3] = o.w;
        }
    }
    // No CTA of a cluster may exit while another still reads its shared memory.
    if (CL > 1)
        cluster_sync();
}

// Merge of two (max, sum) states with the online-softmax rule; maxima are in
// log2 units (already multiplied by log2 e).
__device__ __forceinline__ void merge_state(float &m, float &l, float m2, float l2)
{
    const float mn = fmaxf(m, m2);
    if (mn == -INFINITY)
        return;  // both empty
    l = l * ptx::ex2(m - mn) + l2 * ptx::ex2(m2 - mn);
    m = mn;
}

// Rows too long to keep on chip: pass 1 streams the row once and keeps a running
// (max, sum) per thread, updated element by element; the block merges the
// per-thread states; pass 2 streams the row again and writes the result.
template <int CTA>
__global__ void __launch_bounds__(CTA) softmax_rows_twopass_kernel(const float *x, float *y,
                                                                  int64_t rows, int64_t N)
{
    constexpr int kWarps = CTA / 32;
    __shared__ float sm_m[kWarps], sm_l[kWarps];
    const int64_t row = blockIdx.x;
    if (row >= rows)
        return;
    const float *xr = x + row * N;
    float *yr = y + row * N;

    float m = -INFINITY, l = 0.f;  // m in log2 units
    for (int64_t j = threadIdx.x; j < N; j += CTA) {
        const float t = xr[j] * kLog2e;
        if (t > m) {
            l = l * ptx::ex2(m - t) + 1.f;
            m = t;
        } else if (t != -INFINITY) {  // -inf adds 0 (and -inf - -inf is undefined)
            l += ptx::ex2(t - m);
        }
    }
    for (int o = 16; o > 0; o >>= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
        const float l2 = __shfl_xor_sync(0xffffffffu, l, o);
        merge_state(m, l, m2, l2);
    }
    if ((threadIdx.x & 31) == 0) {
        sm_m[threadIdx.x >> 5] = m;
        sm_l[threadIdx.x >> 5] = l;
    }
    __syncthreads();
    m = sm_m[0];
    l = sm_l[0];
    for (int w = 1; w < kWarps; ++w)
        merge_state(m, l, sm_m[w], sm_l[w]);

    const float inv = __frcp_rn(l);
    for (int64_t j = threadIdx.x; j < N; j += CTA)
        yr[j] = ptx::ex2(fmaf(xr[j], kLog2e, -m)) * inv;
}

template <int G, int V, int CTA, int CL, bool VEC>
cudaError_t launch_resident(const float *x, float *y, int64_t rows, int64_t N,
                            cudaStream_t stream)
{
    auto kern = softmax_rows_kernel<G, V, CTA, CL, VEC>;
    int64_t blocks;
    if (G <= 32)
        blocks = (rows + (CTA / G) - 1) / (CTA / G);
    else
        blocks = rows * CL;
    if (blocks > 0x7fffffffLL)
        return cudaErrorInvalidConfiguration;
    if (CL == 1) {
        kern<<<dim3(unsigned(blocks)), dim3(CTA), 0, stream>>>(x, y, rows, N);
        return cudaGetLastError();
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(blocks));
    cfg.blockDim = dim3(CTA);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CL;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, x, y, rows, N);
}

template <bool VEC>
cudaError_t dispatch(const float *x, float *y, int64_t rows, int64_t N, cudaStream_t stream)
{
    if (N <= 32)     return launch_resident<8, 1, 256, 1, VEC>(x, y, rows, N, stream);
    if (N <= 64)     return launch_resident<16, 1, 256, 1, VEC>(x, y, rows, N, stream);
    if (N <= 128)    return launch_resident<32, 1, 256, 1, VEC>(x, y, rows, N, stream);
    if (N <= 256)    return launch_resident<32, 2, 256, 1, VEC>(x, y, rows, N, stream);
    if (N <= 512)    return launch_resident<32, 4, 256, 1, VEC>(x, y, rows, N, stream);
    if (N <= 1024)   return launch_resident<32, 8, 256, 1, VEC>(x, y, rows, N, stream);
    if (N <= 2048)   return launch_resident<256, 2, 256, 1, VEC>(x, y, rows, N, stream);
    if (N <= 4096)   return launch_resident<256, 4, 256, 1, VEC>(x, y, rows, N, stream);
    if (N <= 8192)   return launch_resident<512, 4, 512, 1, VEC>(x, y, rows, N, stream);
    if (N <= 16384)  return launch_resident<512, 8, 512, 1, VEC>(x, y, rows, N, stream);
    if (N <= 32768)  return launch_resident<1024, 8, 1024, 1, VEC>(x, y, rows, N, stream);
    if (N <= 65536)  return launch_resident<1024, 8, 1024, 2, VEC>(x, y, rows, N, stream);
    if (N <= 131072) return launch_resident<1024, 8, 1024, 4, VEC>(x, y, rows, N, stream);
    if (rows > 0x7fffffffLL)
        return cudaErrorInvalidConfiguration;
    softmax_rows_twopass_kernel<1024><<<dim3(unsigned(rows)), dim3(1024), 0, stream>>>(x, y, rows,
                                                                                     N);
    return cudaGetLastError();
}

}  // namespace

int launch_softmax_rows(const float *x, float *y, int64_t rows, int64_t N, cudaStream_t stream)
{
    if (rows == 0 || N == 0)
        return FA_OK;
    const bool vec = (N % 4 == 0) && (reinterpret_cast<uintptr_t>(x) % 16 == 0) &&
                     (reinterpret_cast<uintptr_t>(y) % 16 == 0);
    cudaError_t e = vec ? dispatch<true>(x, y, rows, N, stream)
                        : dispatch<false>(x, y, rows, N, stream);
    if (e == cudaErrorInvalidConfiguration)
        return FA_ERR_TOO_LARGE;
    return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // namespace fa
