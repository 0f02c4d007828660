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
// Two launches: fp8_qk_mma_kernel (Q, K tiles: the rotation as a tensor-core
// product with fp32 accumulation; V tile amax) and fp8_vt_kernel.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/fa.h"
#include "fa_error.cuh"
#include "launch.h"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr int kRows = 128;          // rows per tile
constexpr float kE4M3Max = 448.f;

__device__ __forceinline__ float warp_max(float v)
{
    for (int o = 16; o > 0; o >>= 1)
        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// ---------------------------------------------------------------------------
// Q and K: X M on the tensor cores, then blockwise e4m3; V: tile amax.
// A persistent kernel, one CTA per SM, walking the work items (tensor, sequence
// * head, 128-row tile) in steps of the grid size:
//   * M' = diag(signs) H_d holds only +-1, exact in bf16, so the tcgen05
//     product X M' (bf16 operands, fp32 accumulation in TMEM) is the rotation
//     before its 1 / sqrt(d).  The epilogue warps write M' into shared memory
//     once (K-major, 128-byte swizzle).
//   * warp 0 streams the X tiles through a 4-stage TMA ring (4-D tensor maps
//     over [B, N, H, d]: rows past a sequence's end read as zero);
//   * warp 1 issues the eight K = 16 MMAs of a Q or K tile into one of two
//     TMEM accumulators; their completion frees the ring stage;
//   * warps 2-5 (one thread per row) read an accumulator twice -- once for
//     the tile amax, once to form the codes -- and send the codes out of one
//     of two shared-memory staging tiles with a TMA store (rows past the end
//     of a sequence are not written); for a V tile they take its amax from
//     the ring stage directly and free the stage.
// ---------------------------------------------------------------------------
constexpr int kQkStages = 4;
constexpr int kQkThreads = 192;
constexpr int kWarpProd = 0, kWarpMmaQ = 1, kEpiWarp0 = 2;
constexpr int kEpiThreads = 128;
constexpr uint32_t kChunk = kRows * 128;      // 128 rows x 128 bytes
constexpr uint32_t kStageBytes = 2 * kChunk;  // one bf16 tile (d = 128)
constexpr uint32_t kOffH = 0;                 // M' (2 chunks)
constexpr uint32_t kOffRing = kOffH + 2 * kChunk;
constexpr uint32_t kOffOut = kOffRing + kQkStages * kStageBytes;   // 2 staging tiles
constexpr uint32_t kOffSgn = kOffOut + 2 * kChunk;   // sign bits of the 16 eight-column units
constexpr uint32_t kOffRed = kOffSgn + 256;          // 2 x 4 warp maxima
constexpr uint32_t kOffBar = kOffRed + 32;
constexpr int kQkBars = 2 * kQkStages + 5;           // full, empty, acc_full[2], acc_empty[2], drain
constexpr uint32_t kOffSlot = kOffBar + 8 * kQkBars; // TMEM base, abort flag
constexpr uint32_t kQkSmemBytes = kOffSlot + 8 + 1024;
constexpr uint32_t kQkTmemCols = 256;                // two 128-column accumulators
static_assert(kQkSmemBytes <= 227 * 1024, "shared memory");

struct QkMmaParams {
    // dense: 4-D maps over [B, N, H, 128], boxes {64, 1, 128, 1} (bf16) and
    // {128, 1, 128, 1} (e4m3); packed: 3-D maps over [total, H, 128], boxes
    // {64, 1, 128} and {128, 1, 128}
    CUtensorMap tm_x[3];              // Q, K, V (bf16)
    CUtensorMap tm_f[2];              // Q', K' (e4m3)
    const float *signs;               // [128], +-1
    float *sq, *sk, *vamax;           // [B, H, n_tiles]
    uint8_t *Qf, *Kf;                 // packed: the codes' rows, for ragged tiles
    const int32_t *cu_seqlens;        // packed: [B + 1] prefix sums (else nullptr)
    int H, n_tiles, BH, n_items;
    int *err_word;
};

// A warp's wait: lane 0 polls (bounded) and shares the outcome.
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, volatile int *abort,
                                          int *err_word)
{
    int ok = 1;
    if ((threadIdx.x & 31) == 0)
        ok = ptx::mbar_wait(bar, parity, abort, err_word) ? 1 : 0;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    __syncwarp();
    return ok != 0;
}

// Bounded wait for a barrier phase before the CTA leaves after an abort, so
// that no copy or product in flight still targets its shared or tensor memory.
__device__ __forceinline__ void drain(uint64_t *bar, uint32_t parity)
{
    const uint64_t t0 = ptx::globaltimer();
    for (uint32_t it = 0; it < kWaitMaxPolls; ++it) {
        if (ptx::mbar_try_wait(bar, parity))
            return;
        if ((it & 255u) == 255u && ptx::globaltimer() - t0 > kWaitTimeoutNs)
            return;
    }
}

struct Item {
    int which, b, h, tile;
    int64_t sidx;                     // (b * H + h) * n_tiles + tile
    int64_t row0;                     // packed: the tile's first row of [total, H, d]
    int valid;                        // rows of the tile inside the sequence (<= 0: none)
};
template <bool PACKED>
__device__ __forceinline__ Item decode_item(const QkMmaParams &p, int j)
{
    Item it;
    it.tile = j % p.n_tiles;
    const int r = j / p.n_tiles;
    const int bh = r % p.BH;
    it.which = r / p.BH;
    it.b = bh / p.H;
    it.h = bh % p.H;
    it.sidx = int64_t(bh) * p.n_tiles + it.tile;
    it.row0 = 0;
    it.valid = kRows;                 // dense: the 4-D maps clip the sequence's end
    if constexpr (PACKED) {
        const int64_t s0 = p.cu_seqlens[it.b], s1 = p.cu_seqlens[it.b + 1];
        it.row0 = s0 + int64_t(it.tile) * kRows;
        const int64_t v = s1 - it.row0;
        it.valid = v < kRows ? int(v) : kRows;
    }
    return it;
}

// PACKED: sequences from cu_seqlens over [total, H, d] (3-D maps); the dense
// instantiation keeps the 4-D maps and whole-tile stores.
template <bool PACKED>
__global__ void __launch_bounds__(kQkThreads, 1) fp8_qk_mma_kernel(const __grid_constant__ QkMmaParams p)
{
    constexpr int D = 128;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *hs = smem + kOffH, *ring = smem + kOffRing, *out = smem + kOffOut;
    uint32_t *sgn = reinterpret_cast<uint32_t *>(smem + kOffSgn);
    float *red = reinterpret_cast<float *>(smem + kOffRed);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kOffBar);
    uint64_t *full = bars, *empty = bars + kQkStages;
    uint64_t *acc_full = bars + 2 * kQkStages, *acc_empty = acc_full + 2, *drain_bar = acc_full + 4;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kOffSlot);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kQkStages; ++s) {
            ptx::mbar_init(&full[s], 1);
            ptx::mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            ptx::mbar_init(&acc_full[a], 1);
            ptx::mbar_init(&acc_empty[a], kEpiThreads / 32);
        }
        ptx::mbar_init(drain_bar, 1);
        *abort_flag = 0;
        ptx::fence_barrier_init();
    }
    if (warp == kWarpMmaQ) {
        ptx::tmem_alloc(tmem_slot, kQkTmemCols);
        ptx::tmem_relinquish();
    }
    // sign bits of M' rows: word t covers columns 2t (bit 15) and 2t + 1 (bit
    // 31), the sign positions of a bf16 pair
    if (threadIdx.x < D / 2) {
        const int k = 2 * int(threadIdx.x);
        sgn[threadIdx.x] =
            (p.signs[k] < 0.f ? 0x8000u : 0u) | (p.signs[k + 1] < 0.f ? 0x80000000u : 0u);
    }
    ptx::tc_fence_before_sync();
    __syncthreads();
    ptx::tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    if (warp == kWarpProd) {
        // ======================= TMA producer ==============================
        if (lane == 0) {
            int last_phase[kQkStages];
            for (int s = 0; s < kQkStages; ++s)
                last_phase[s] = -1;
            int stage = 0;
            uint32_t phase = 0;
            for (int j = int(blockIdx.x); j < p.n_items; j += int(gridDim.x)) {
                const Item it = decode_item<PACKED>(p, j);
                if (it.valid <= 0)
                    continue;                      // a tile past its sequence's end
                if (!ptx::mbar_wait(&empty[stage], phase ^ 1u, abort_flag, p.err_word))
                    break;
                uint8_t *dst = ring + stage * kStageBytes;
                ptx::mbar_arrive_expect_tx(&full[stage], kStageBytes);
                if constexpr (PACKED) {
                    // rows past the sequence's end are the next one's: the
                    // epilogue leaves them out of the amax and does not store them
                    ptx::tma_load_3d(dst, &p.tm_x[it.which], &full[stage], 0, it.h,
                                     int(it.row0));
                    ptx::tma_load_3d(dst + kChunk, &p.tm_x[it.which], &full[stage], 64, it.h,
                                     int(it.row0));
                } else {
                    ptx::tma_load_4d(dst, &p.tm_x[it.which], &full[stage], 0, it.h,
                                     it.tile * kRows, it.b);
                    ptx::tma_load_4d(dst + kChunk, &p.tm_x[it.which], &full[stage], 64, it.h,
                                     it.tile * kRows, it.b);
                }
                last_phase[stage] = int(phase);
                if (++stage == kQkStages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (*abort_flag)
                for (int s = 0; s < kQkStages; ++s)
                    if (last_phase[s] >= 0)
                        drain(&full[s], uint32_t(last_phase[s]));
        }
        __syncwarp();
    } else if (warp == kWarpMmaQ) {
        // ======================= MMA issuer (whole warp) =====================
        asm volatile("bar.sync 2, %0;" ::"n"(32 + kEpiThreads) : "memory");   // M' written
        constexpr uint32_t idesc = ptx::idesc_bf16_f32(kRows, D, false);
        constexpr uint64_t desc_kmajor = ptx::smem_desc_base(16, 1024);
        const uint64_t db = ptx::smem_desc(desc_kmajor, ptx::smem_u32(hs));
        const uint64_t dring = ptx::smem_desc(desc_kmajor, ptx::smem_u32(ring));
        int stage = 0, abuf = 0;
        uint32_t phase = 0, aphase = 0;
        for (int j = int(blockIdx.x); j < p.n_items; j += int(gridDim.x)) {
            const Item itm = decode_item<PACKED>(p, j);
            if (itm.valid <= 0)
                continue;                          // skipped by every role alike
            const int which = itm.which;
            const int st = stage;
            const uint32_t ph = phase;
            if (++stage == kQkStages) {
                stage = 0;
                phase ^= 1u;
            }
            if (which == 2)
                continue;                          // V tiles: no product
            if (!ptx::mbar_wait_warp(&full[st], ph, abort_flag, p.err_word) ||
                !ptx::mbar_wait_warp(&acc_empty[abuf], aphase ^ 1u, abort_flag, p.err_word))
                break;
            ptx::tc_fence_after_sync();
            const uint64_t da = dring + ((st * kStageBytes) >> 4);
            if (ptx::elect_one()) {
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint64_t off = ((kk >> 2) * kChunk + (kk & 3) * 32) >> 4;
                    ptx::mma_ss(tmem + uint32_t(abuf) * 128, da + off, db + off, idesc,
                                kk > 0 ? 1u : 0u);
                }
                ptx::mma_commit(&empty[st]);
                ptx::mma_commit(&acc_full[abuf]);
            }
            __syncwarp();
            if (++abuf == 2) {
                abuf = 0;
                aphase ^= 1u;
            }
        }
        if (ptx::elect_one()) {
            ptx::mma_commit(drain_bar);
            drain(drain_bar, 0);
        }
        __syncwarp();
    } else {
        // ======================= epilogue (one thread per row) ===============
        const int et = int(threadIdx.x) - kEpiWarp0 * 32;    // 0 .. 127
        const int q = warp & 3;                  // TMEM lane quarter of this warp
        const int r = q * 32 + lane;             // tile row = TMEM lane
        // M' row n = et, K-major with the 128-byte swizzle (16-byte unit u of
        // row n at unit u ^ (n % 8)): entry (n, k) = sign_k (-1)^popc(n & k).
        // For the 8 columns k0 + t of a unit (k0 a multiple of 8) the
        // Hadamard sign splits as (-1)^popc(n & k0) (-1)^popc(n & t).
        {
            const uint32_t n = uint32_t(et);
            uint32_t tpl[4];
#pragma unroll
            for (int j = 0; j < 4; ++j)
                tpl[j] = 0x3F803F80u | ((uint32_t(__popc(n & uint32_t(2 * j))) & 1u) << 15) |
                         ((uint32_t(__popc(n & uint32_t(2 * j + 1))) & 1u) << 31);
#pragma unroll
            for (int v = 0; v < 16; ++v) {
                const uint32_t flip = (uint32_t(__popc(n & uint32_t(8 * v))) & 1u) * 0x80008000u;
                const uint4 sg = *reinterpret_cast<const uint4 *>(sgn + 4 * v);
                uint4 w;
                w.x = tpl[0] ^ sg.x ^ flip;
                w.y = tpl[1] ^ sg.y ^ flip;
                w.z = tpl[2] ^ sg.z ^ flip;
                w.w = tpl[3] ^ sg.w ^ flip;
                *reinterpret_cast<uint4 *>(hs + (v >> 3) * kChunk + n * 128 +
                                           (((v & 7) ^ (n & 7)) << 4)) = w;
            }
        }
        ptx::fence_proxy_async_smem();         // M' -> the tensor cores' reads
        asm volatile("bar.sync 2, %0;" ::"n"(32 + kEpiThreads) : "memory");

        const float inv_d = rsqrtf(float(D));
        const uint32_t lane_bits = uint32_t(q * 32) << 16;
        int stage = 0, abuf = 0, ob = 0, ib = 0;
        uint32_t phase = 0, aphase = 0;
        for (int j = int(blockIdx.x); j < p.n_items; j += int(gridDim.x)) {
            const Item it = decode_item<PACKED>(p, j);
            if (it.valid <= 0)
                continue;                          // skipped by every role alike
            const bool row_in = !PACKED || r < it.valid;   // this thread's row is in the sequence
            const int st = stage;
            const uint32_t ph = phase;
            if (++stage == kQkStages) {
                stage = 0;
                phase ^= 1u;
            }
            float *rd = red + 4 * ib;            // this item's warp maxima
            ib ^= 1;
            if (it.which == 2) {
                // V: the tile's amax, a max of |bf16| values (exact in bf16);
                // the row's 16-byte units are visited in swizzled order so
                // that a warp's loads fall in distinct banks
                const bool ok = warp_wait(&full[st], ph, abort_flag, p.err_word);
                uint32_t m = 0;                  // two |bf16| maxima, as bf16x2
                if (ok && row_in) {
                    const uint8_t *src = ring + st * kStageBytes;
#pragma unroll
                    for (int c = 0; c < 2; ++c)
#pragma unroll
                        for (int u = 0; u < 8; ++u) {
                            const uint4 w = *reinterpret_cast<const uint4 *>(
                                src + c * kChunk + r * 128 + ((u ^ (r & 7)) << 4));
                            const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const __nv_bfloat162 a = __hmax2(
                                    *reinterpret_cast<const __nv_bfloat162 *>(&m),
                                    __habs2(*reinterpret_cast<const __nv_bfloat162 *>(&ww[e])));
                                m = *reinterpret_cast<const uint32_t *>(&a);
                            }
                        }
                }
                const __nv_bfloat162 mm = *reinterpret_cast<const __nv_bfloat162 *>(&m);
                const float amax = warp_max(fmaxf(__low2float(mm), __high2float(mm)));
                if (lane == 0)
                    rd[q] = amax;
                // the 128 threads agree on leaving (a wait given up in any warp)
                if (ptx::bar_red_or(1, kEpiThreads, !ok))
                    break;
                if (et == 0) {
                    p.vamax[it.sidx] = fmaxf(fmaxf(rd[0], rd[1]), fmaxf(rd[2], rd[3]));
                    ptx::mbar_arrive(&empty[st]);    // every row has been read
                }
                continue;
            }
            const bool ok = warp_wait(&acc_full[abuf], aphase, abort_flag, p.err_word);
            const uint32_t t_row = tmem + lane_bits + uint32_t(abuf) * 128;
            // pass 1: the tile amax of the rotated rows (|s| / sqrt(d) is
            // monotone in |s|, so the scaling moves outside the max)
            float amax = 0.f;
            if (ok) {
                ptx::tc_fence_after_sync();
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t v[32];
                    ptx::tmem_ld32(t_row + 32 * c, v);
                    ptx::tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; e += 2)
                        amax = ptx::max3(amax, fabsf(__uint_as_float(v[e])),
                                         fabsf(__uint_as_float(v[e + 1])));
                }
                if (!row_in)
                    amax = 0.f;                  // a row of the next sequence
            }
            amax = warp_max(amax) * inv_d;
            if (lane == 0)
                rd[q] = amax;
            if (et == 0)                         // the staging tile's last store has read it
                asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
            if (ptx::bar_red_or(1, kEpiThreads, !ok))
                break;
            amax = fmaxf(fmaxf(rd[0], rd[1]), fmaxf(rd[2], rd[3]));
            const float scale = amax > 0.f ? amax / kE4M3Max : 1.f;
            if (et == 0)
                (it.which == 0 ? p.sq : p.sk)[it.sidx] = scale;
            const float mul = inv_d * (1.f / scale);
            // pass 2: the codes of row r into staging tile ob, or, for a
            // packed tile cut by its sequence's end, straight to its row
            const bool ragged = PACKED && it.valid < kRows;
            uint8_t *row = out + ob * kChunk + r * 128;
            uint8_t *grow = (it.which == 0 ? p.Qf : p.Kf) + ((it.row0 + r) * p.H + it.h) * D;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t v[32];
                ptx::tmem_ld32(t_row + 32 * c, v);
                ptx::tmem_wait_ld();
                uint32_t w[8];
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    w[k] = ptx::pack_e4m3x4(__uint_as_float(v[4 * k]) * mul,
                                            __uint_as_float(v[4 * k + 1]) * mul,
                                            __uint_as_float(v[4 * k + 2]) * mul,
                                            __uint_as_float(v[4 * k + 3]) * mul);
                if (ragged) {
                    if (row_in) {
                        *reinterpret_cast<uint4 *>(grow + 32 * c) = make_uint4(w[0], w[1], w[2], w[3]);
                        *reinterpret_cast<uint4 *>(grow + 32 * c + 16) =
                            make_uint4(w[4], w[5], w[6], w[7]);
                    }
                    continue;
                }
                *reinterpret_cast<uint4 *>(row + (((2 * c) ^ (r & 7)) << 4)) =
                    make_uint4(w[0], w[1], w[2], w[3]);
                *reinterpret_cast<uint4 *>(row + (((2 * c + 1) ^ (r & 7)) << 4)) =
                    make_uint4(w[4], w[5], w[6], w[7]);
            }
            ptx::tc_fence_before_sync();
            __syncwarp();
            if (lane == 0)
                ptx::mbar_arrive(&acc_empty[abuf]);  // this warp's accumulator rows are read
            ptx::fence_proxy_async_smem();       // staged codes -> the TMA store
            asm volatile("bar.sync 1, %0;" ::"n"(kEpiThreads) : "memory");
            if (et == 0 && !ragged) {
                if constexpr (PACKED)
                    ptx::tma_store_3d(&p.tm_f[it.which], out + ob * kChunk, 0, it.h,
                                      int(it.row0));
                else
                    ptx::tma_store_4d(&p.tm_f[it.which], out + ob * kChunk, 0, it.h,
                                      it.tile * kRows, it.b);
                asm volatile("cp.async.bulk.commit_group;" ::: "memory");
            }
            ob ^= 1;
            if (++abuf == 2) {
                abuf = 0;
                aphase ^= 1u;
            }
        }
        if (et == 0)
            asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
    }
    ptx::tc_fence_before_sync();
    __syncthreads();
    if (warp == kWarpMmaQ) {
        ptx::tc_fence_after_sync();
        ptx::tmem_dealloc(tmem, kQkTmemCols);
    }
}

struct VtParams {
    CUtensorMap tm_vt;                // Vt: e4m3 [B*H*d, n_pad], box {128 keys, 128 rows}
    const __nv_bfloat16 *V;           // dense [B, N, H, d]; packed [total, H, d]
    const float *vamax;               // [B, H, n_tiles]
    float *sv;                        // [B, H]
    const int32_t *cu_seqlens;        // packed: [B + 1] prefix sums (else nullptr)
    int B, H, N, n_tiles;
};

constexpr uint32_t kVtSmemBytes = kRows * 128 + 1024;

// V' = codes of V / sv, transposed per head ([B, H, d, n_pad]; keys past N are
// zero codes).  One CTA (8 warps) per (sequence * head, 128-key tile): lane l
// takes keys 4l .. 4l + 3 and warp w head-dim columns 16w .. 16w + 15 (two
// 16-byte pieces of a key row, one 32-byte sector).  For each of its columns
// a lane writes the codes of its 4 keys as one 32-bit word into the staging
// tile (rows = columns, 128-byte swizzle: the 32 lanes' words of one column
// fall in distinct banks), and one TMA store sends the tile.
__global__ void __launch_bounds__(256) fp8_vt_kernel(const __grid_constant__ VtParams p)
{
    constexpr int D = 128;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *stage = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int bh = blockIdx.x, tile = blockIdx.y;
    const int b = bh / p.H, h = bh % p.H;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int c0 = 16 * warp;
    // the sequence's first row and length (packed: from the prefix sums);
    // tiles past its end are never read by the attention kernel
    int64_t row0 = int64_t(b) * p.N;
    int L = p.N;
    if (p.cu_seqlens != nullptr) {
        row0 = p.cu_seqlens[b];
        L = int(p.cu_seqlens[b + 1] - row0);
    }
    if (tile * kRows >= L)
        return;
    const int n_tiles = (L + kRows - 1) / kRows;
    // the tile's loads go out first, then the per-head amax (one tile amax per
    // lane, reduced across the warp), then the conversions
    uint4 raw[4][2];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int key = tile * kRows + 4 * lane + j;
        if (key < L) {
            const uint4 *src = reinterpret_cast<const uint4 *>(
                p.V + ((row0 + key) * p.H + h) * D + c0);
            raw[j][0] = src[0];
            raw[j][1] = src[1];
        } else {
            raw[j][0] = make_uint4(0, 0, 0, 0);
            raw[j][1] = make_uint4(0, 0, 0, 0);
        }
    }
    // Launched as a programmatic dependent of the quantisation kernel: V (an
    // input) is loaded above; the per-tile amax it wrote is read only after
    // the wait, which returns once that kernel has completed.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    float amax = 0.f;
    for (int t = lane; t < n_tiles; t += 32)
        amax = fmaxf(amax, p.vamax[int64_t(bh) * p.n_tiles + t]);
    amax = warp_max(amax);
    const float scale = amax > 0.f ? amax / kE4M3Max : 1.f;
    if (tile == 0 && threadIdx.x == 0)
        p.sv[bh] = scale;
    const float inv = 1.f / scale;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        float f[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint4 u = raw[j][i >> 3];
            const int e = i & 7;
            const uint32_t w = (e >> 1) == 0 ? u.x : (e >> 1) == 1 ? u.y : (e >> 1) == 2 ? u.z : u.w;
            f[j] = __uint_as_float((e & 1) ? (w & 0xffff0000u) : (w << 16)) * inv;
        }
        const int c = c0 + i;
        *reinterpret_cast<uint32_t *>(stage + c * 128 + (((lane >> 2) ^ (c & 7)) << 4) +
                                      (lane & 3) * 4) = ptx::pack_e4m3x4(f[0], f[1], f[2], f[3]);
    }
    ptx::fence_proxy_async_smem();             // staged codes -> the TMA store
    __syncthreads();
    if (threadIdx.x == 0) {
        ptx::tma_store_2d(&p.tm_vt, stage, tile * kRows, bh * D);
        ptx::bulk_commit_and_wait_read();
    }
}

}  // namespace

int launch_fp8_quantize(const Fp8QuantArgs &a, cudaStream_t stream)
{
    if (a.d != 128)
        return FA_ERR_UNSUPPORTED;
    const int n_tiles = (a.N + kRows - 1) / kRows;
    // work items of the first kernel are counted in an int; the second
    // kernel's grid takes the tiles of a head along y (at most 65535)
    if (3 * int64_t(a.B) * a.H * n_tiles > 0x7fffffffLL || n_tiles > 65535)
        return FA_ERR_TOO_LARGE;
    QkMmaParams q;
    if (a.cu_seqlens != nullptr) {
        if (!make_tmap_bf16(&q.tm_x[0], a.Q, a.total, a.H, a.d) ||
            !make_tmap_bf16(&q.tm_x[1], a.K, a.total, a.H, a.d) ||
            !make_tmap_bf16(&q.tm_x[2], a.V, a.total, a.H, a.d) ||
            !make_tmap_e4m3_rows(&q.tm_f[0], a.Qf, a.total, a.H, a.d) ||
            !make_tmap_e4m3_rows(&q.tm_f[1], a.Kf, a.total, a.H, a.d))
            return FA_ERR_CUDA;
    } else if (!make_tmap_seq_4d(&q.tm_x[0], a.Q, false, a.B, a.N, a.H, a.d) ||
               !make_tmap_seq_4d(&q.tm_x[1], a.K, false, a.B, a.N, a.H, a.d) ||
               !make_tmap_seq_4d(&q.tm_x[2], a.V, false, a.B, a.N, a.H, a.d) ||
               !make_tmap_seq_4d(&q.tm_f[0], a.Qf, true, a.B, a.N, a.H, a.d) ||
               !make_tmap_seq_4d(&q.tm_f[1], a.Kf, true, a.B, a.N, a.H, a.d)) {
        return FA_ERR_CUDA;
    }
    q.Qf = a.Qf;
    q.Kf = a.Kf;
    q.cu_seqlens = a.cu_seqlens;
    q.signs = a.signs;
    q.sq = a.sq;
    q.sk = a.sk;
    q.vamax = a.vamax;
    q.H = a.H;
    q.n_tiles = n_tiles;
    q.BH = a.B * a.H;
    q.n_items = 3 * q.BH * n_tiles;
    q.err_word = a.err_word;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        sms <= 0)
        return FA_ERR_CUDA;
    static PerDeviceOnce once_qk, once_qk_packed;
    const bool packed = a.cu_seqlens != nullptr;
    auto kqk = packed ? fp8_qk_mma_kernel<true> : fp8_qk_mma_kernel<false>;
    if (!set_max_dynamic_smem(packed ? once_qk_packed : once_qk,
                              reinterpret_cast<const void *>(kqk), int(kQkSmemBytes)))
        return FA_ERR_CUDA;
    const int grid = q.n_items < sms ? q.n_items : sms;
    kqk<<<grid, kQkThreads, kQkSmemBytes, stream>>>(q);
    if (cudaGetLastError() != cudaSuccess)
        return FA_ERR_CUDA;
    VtParams v;
    if (!make_tmap_e4m3_vt(&v.tm_vt, a.Vt, int64_t(a.B) * a.H * a.d, int64_t(n_tiles) * kRows,
                           a.d))
        return FA_ERR_CUDA;
    v.V = static_cast<const __nv_bfloat16 *>(a.V);
    v.vamax = a.vamax;
    v.sv = a.sv;
    v.cu_seqlens = a.cu_seqlens;
    v.B = a.B;
    v.H = a.H;
    v.N = a.N;
    v.n_tiles = n_tiles;
    static PerDeviceOnce once_vt;
    if (!set_max_dynamic_smem(once_vt, reinterpret_cast<const void *>(fp8_vt_kernel),
                              int(kVtSmemBytes)))
        return FA_ERR_CUDA;
    // programmatic dependent launch: its launch and its loads of V overlap
    // the end of the quantisation kernel
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(a.B * a.H), unsigned(n_tiles));
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = kVtSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, fp8_vt_kernel, v) != cudaSuccess)
        return FA_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // namespace fa
