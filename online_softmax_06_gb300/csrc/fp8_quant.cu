// fp8_quant.cu -- the quantisation pass of the FP8 attention forward
// ("少搬一趟：FlashAttention 四代进化史" §4.6: blockwise quantisation and
// incoherent processing).
//
//   * Q and K rows are multiplied by M = diag(signs) H_d / sqrt(d) (random +-1
//     signs, the Sylvester-Hadamard matrix), so (QM)(KM)^T = Q K^T while large
//     components are spread over the row; each 128-row tile of a head then gets
//     its own scale amax / 448 and its values become e4m3 codes (round to
//     nearest even, saturating).
//   * V gets one scale per (sequence, head) and is written transposed per head
//     ([B, H, d, Npad] e4m3), so that the P V product can read it as a K-major
//     operand (keys contiguous).
// Two launches: fp8_qk_kernel (Q, K tiles; V tile amax) and fp8_vt_kernel.
// The products run in fp32: bf16 inputs, the rotation in registers with warp
// shuffles (a fast Walsh-Hadamard transform: log2 d butterfly stages).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <type_traits>

#include "../../include/fa.h"
#include "launch.h"

namespace fa {
namespace {

constexpr int kRows = 128;          // rows per tile
// 32 warps of 4 rows each, two CTAs per SM (32 registers a thread): loads of
// one CTA overlap the other's arithmetic; the rows stay in registers
constexpr int kWarps = 32;
constexpr float kE4M3Max = 448.f;

__device__ __forceinline__ float warp_max(float v)
{
    for (int o = 16; o > 0; o >>= 1)
        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// Two floats to two e4m3 codes (round to nearest even, saturating): `lo` in
// bits 0..7, `hi` in bits 8..15.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi)
{
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// In-place x M for one row held by a warp: lane l holds elements l*E .. l*E+E-1
// (E = D / 32).  Butterfly stage b pairs element i with i ^ (1 << b); the lower
// index keeps a + b, the upper a - b.
template <int D>
__device__ __forceinline__ void rotate_row(float (&x)[D / 32], const float (&sg)[D / 32], int lane)
{
    constexpr int E = D / 32;
    constexpr int LE = (E == 4) ? 2 : 1;
#pragma unroll
    for (int k = 0; k < E; ++k)
        x[k] *= sg[k];
#pragma unroll
    for (int b = 0; b < LE; ++b) {                 // partners within the lane
#pragma unroll
        for (int k = 0; k < E; ++k)
            if ((k & (1 << b)) == 0) {
                const float u = x[k], v = x[k | (1 << b)];
                x[k] = u + v;
                x[k | (1 << b)] = u - v;
            }
    }
#pragma unroll
    for (int b = 0; b < 5; ++b) {                  // partners in other lanes
        // the lower lane keeps x + y, the upper y - x: fma(x, +-1, y)
        const float sgn = ((lane >> b) & 1) ? -1.f : 1.f;
#pragma unroll
        for (int k = 0; k < E; ++k) {
            const float y = __shfl_xor_sync(0xffffffffu, x[k], 1 << b);
            x[k] = fmaf(x[k], sgn, y);
        }
    }
    const float inv = rsqrtf(float(D));
#pragma unroll
    for (int k = 0; k < E; ++k)
        x[k] *= inv;
}

struct QuantParams {
    const __nv_bfloat16 *Q, *K, *V;
    const float *signs;               // [d], +-1
    uint8_t *Qf, *Kf;                 // [B*N, H, d] e4m3
    float *sq, *sk, *vamax;           // [B, H, n_tiles]
    int B, H, N, n_tiles;
};

// blockIdx: x = tile, y = b * H + h, z = 0 (Q), 1 (K), 2 (V amax only).
template <int D>
__global__ void __launch_bounds__(kWarps * 32, 2) fp8_qk_kernel(const QuantParams p)
{
    constexpr int E = D / 32;
    constexpr int kRowsPerWarp = kRows / kWarps;
    __shared__ float red[kWarps];
    const int tile = blockIdx.x, bh = blockIdx.y, which = blockIdx.z;
    const int b = bh / p.H, h = bh % p.H;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const __nv_bfloat16 *src = which == 0 ? p.Q : which == 1 ? p.K : p.V;
    float sg[E];
#pragma unroll
    for (int k = 0; k < E; ++k)
        sg[k] = p.signs[lane * E + k];

    float x[kRowsPerWarp][E];
    // every row's load is issued before any arithmetic
    using Raw = typename std::conditional<E == 4, uint2, uint32_t>::type;
    Raw raw[kRowsPerWarp];
#pragma unroll
    for (int rr = 0; rr < kRowsPerWarp; ++rr) {
        const int row = tile * kRows + warp * kRowsPerWarp + rr;
        const __nv_bfloat16 *rp = src + ((int64_t(b) * p.N + row) * p.H + h) * D + lane * E;
        raw[rr] = row < p.N ? *reinterpret_cast<const Raw *>(rp) : Raw{};
    }
    float amax = 0.f;
#pragma unroll
    for (int rr = 0; rr < kRowsPerWarp; ++rr) {
        if constexpr (E == 4) {
            const uint2 u = raw[rr];
            const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.x));
            const float2 c = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.y));
            x[rr][0] = a.x;
            x[rr][1] = a.y;
            x[rr][2] = c.x;
            x[rr][3] = c.y;
        } else {
            const uint32_t u = raw[rr];
            const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u));
            x[rr][0] = a.x;
            x[rr][1] = a.y;
        }
        if (which < 2)
            rotate_row<D>(x[rr], sg, lane);
#pragma unroll
        for (int k = 0; k < E; ++k)
            amax = fmaxf(amax, fabsf(x[rr][k]));
    }
    amax = warp_max(amax);
    if (lane == 0)
        red[warp] = amax;
    __syncthreads();
    amax = warp_max(red[lane]);             // one partial per warp, 32 warps
    const int64_t sidx = int64_t(bh) * p.n_tiles + tile;
    if (which == 2) {
        if (threadIdx.x == 0)
            p.vamax[sidx] = amax;
        return;
    }
    const float scale = amax > 0.f ? amax / kE4M3Max : 1.f;
    if (threadIdx.x == 0)
        (which == 0 ? p.sq : p.sk)[sidx] = scale;
    const float inv = 1.f / scale;
    uint8_t *dst = which == 0 ? p.Qf : p.Kf;
#pragma unroll
    for (int rr = 0; rr < kRowsPerWarp; ++rr) {
        const int row = tile * kRows + warp * kRowsPerWarp + rr;
        if (row >= p.N)
            continue;
        uint8_t *rp = dst + ((int64_t(b) * p.N + row) * p.H + h) * D + lane * E;
        if constexpr (E == 4) {
            const uint32_t w = e4m3x2(x[rr][0] * inv, x[rr][1] * inv) |
                               (e4m3x2(x[rr][2] * inv, x[rr][3] * inv) << 16);
            *reinterpret_cast<uint32_t *>(rp) = w;
        } else {
            *reinterpret_cast<uint16_t *>(rp) =
                uint16_t(e4m3x2(x[rr][0] * inv, x[rr][1] * inv));
        }
    }
}

struct VtParams {
    const __nv_bfloat16 *V;
    const float *vamax;               // [B, H, n_tiles]
    uint8_t *Vt;                      // [B, H, d, n_pad] e4m3
    float *sv;                        // [B, H]
    int B, H, N, n_tiles, n_pad;
};

// One CTA per (tile, b * H + h): V tile [128 keys][d] -> Vt rows d x 128 keys.
// The tile is transposed through shared memory as e4m3 bytes (row pitch 132:
// the byte writes of a warp and its 32-bit reads fall in distinct banks).
template <int D>
__global__ void __launch_bounds__(256) fp8_vt_kernel(const VtParams p)
{
    constexpr int kPitch = kRows + 4;
    __shared__ __align__(16) uint8_t tileT[D * kPitch];
    const int tile = blockIdx.x, bh = blockIdx.y;
    const int b = bh / p.H, h = bh % p.H;
    float amax = 0.f;
    for (int t = 0; t < p.n_tiles; ++t)
        amax = fmaxf(amax, p.vamax[int64_t(bh) * p.n_tiles + t]);
    const float scale = amax > 0.f ? amax / kE4M3Max : 1.f;
    if (tile == 0 && threadIdx.x == 0)
        p.sv[bh] = scale;
    const float inv = 1.f / scale;
    // load: thread -> (key r, head-dim pair c, c + 1); every load of the
    // thread is issued before the first conversion
    constexpr int kPairs = kRows * D / 2 / 256;       // per thread (256 threads)
    __nv_bfloat162 raw[kPairs];
#pragma unroll
    for (int u = 0; u < kPairs; ++u) {
        const int e = u * 256 + int(threadIdx.x);
        const int r = e / (D / 2), c = (e % (D / 2)) * 2;
        const int row = tile * kRows + r;
        raw[u] = row < p.N ? *reinterpret_cast<const __nv_bfloat162 *>(
                                 p.V + ((int64_t(b) * p.N + row) * p.H + h) * D + c)
                           : __floats2bfloat162_rn(0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < kPairs; ++u) {
        const int e = u * 256 + int(threadIdx.x);
        const int r = e / (D / 2), c = (e % (D / 2)) * 2;
        const uint32_t w = e4m3x2(__low2float(raw[u]) * inv, __high2float(raw[u]) * inv);
        tileT[c * kPitch + r] = uint8_t(w & 0xffu);
        tileT[(c + 1) * kPitch + r] = uint8_t(w >> 8);
    }
    __syncthreads();
    // store: each thread writes 4 keys of one head-dim row (rows of 128 bytes
    // stay contiguous)
    uint8_t *out = p.Vt + (int64_t(bh) * D) * p.n_pad + int64_t(tile) * kRows;
    for (int e = threadIdx.x; e < D * kRows / 4; e += blockDim.x) {
        const int c = e / (kRows / 4), r = (e % (kRows / 4)) * 4;
        *reinterpret_cast<uint32_t *>(out + int64_t(c) * p.n_pad + r) =
            *reinterpret_cast<const uint32_t *>(&tileT[c * kPitch + r]);
    }
}

}  // namespace

int launch_fp8_quantize(const Fp8QuantArgs &a, cudaStream_t stream)
{
    const int n_tiles = (a.N + kRows - 1) / kRows;
    QuantParams q{static_cast<const __nv_bfloat16 *>(a.Q), static_cast<const __nv_bfloat16 *>(a.K),
                  static_cast<const __nv_bfloat16 *>(a.V), a.signs, a.Qf, a.Kf, a.sq, a.sk,
                  a.vamax, a.B, a.H, a.N, n_tiles};
    const dim3 grid(unsigned(n_tiles), unsigned(a.B * a.H), 3);
    if (a.d == 128)
        fp8_qk_kernel<128><<<grid, kWarps * 32, 0, stream>>>(q);
    else
        fp8_qk_kernel<64><<<grid, kWarps * 32, 0, stream>>>(q);
    if (cudaGetLastError() != cudaSuccess)
        return FA_ERR_CUDA;
    VtParams v{static_cast<const __nv_bfloat16 *>(a.V), a.vamax, a.Vt, a.sv, a.B, a.H, a.N,
               n_tiles, n_tiles * kRows};
    const dim3 grid_v(unsigned(n_tiles), unsigned(a.B * a.H));
    if (a.d == 128)
        fp8_vt_kernel<128><<<grid_v, 256, 0, stream>>>(v);
    else
        fp8_vt_kernel<64><<<grid_v, 256, 0, stream>>>(v);
    return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // namespace fa
