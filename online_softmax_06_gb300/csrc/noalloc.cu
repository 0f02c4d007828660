// noalloc.cu -- split-KV attention forward with the library's own static
// scratch, for callers that cannot allocate device memory or hand over a
// workspace (fa_attention_fwd_splitkv_noalloc in include/fa.h).
//
// The partial results of the key splits (fp32 O and lse per split) live in one
// file-scope device array of FA_NOALLOC_SCRATCH_BYTES.  The array sits in this
// translation unit alone, so the CUDA runtime loads it (and its device memory
// is taken) only on devices where this entry point is called, when modules are
// loaded lazily (the CUDA default).  Its address is looked up once per device
// and cached.  Nothing here allocates: the call validates, carves the array
// into O_accum and lse_accum, and hands them to fa_attention_fwd_splitkv.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/fa.h"

static __device__ __align__(256) float g_splitkv_scratch[FA_NOALLOC_SCRATCH_BYTES / sizeof(float)];

namespace fa {
namespace {

constexpr int kMaxDevices = 64;

std::mutex g_scratch_mutex;
float *g_scratch_addr[kMaxDevices] = {};

// Device address of g_splitkv_scratch on the current device, looked up with
// that device current on the first call and cached.
int scratch_on_current_device(float **ptr)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return FA_ERR_NO_DEVICE;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (g_scratch_addr[dev] == nullptr) {
        float *addr = nullptr;
        if (cudaGetSymbolAddress((void **)&addr, g_splitkv_scratch) != cudaSuccess ||
            addr == nullptr)
            return FA_ERR_CUDA;
        g_scratch_addr[dev] = addr;
    }
    *ptr = g_scratch_addr[dev];
    return FA_OK;
}

}  // namespace
}  // namespace fa

extern "C" int fa_attention_fwd_splitkv_noalloc(const void *Q, const void *K, const void *V,
                                                void *O, float *lse, int B, int H, int Nq, int Nk,
                                                int d, float scale, int causal, int num_splits)
{
    // The argument errors fa_attention_fwd_splitkv reports before it looks at
    // the scratch come first, so both functions answer them alike.
    if (B < 0 || H < 0 || Nq < 0 || Nk < 0 || num_splits < 0)
        return FA_ERR_BAD_SIZE;
    if (causal && Nk < Nq)
        return FA_ERR_BAD_SIZE;
    if (d != 64 && d != 128)
        return FA_ERR_UNSUPPORTED;
    if (B == 0 || H == 0 || Nq == 0 || Nk == 0)
        return fa_attention_fwd_splitkv(Q, K, V, O, lse, B, H, Nq, Nk, d, scale, causal, 1,
                                        nullptr, nullptr);

    // the split count fa_attention_fwd_splitkv would use (also checks the device)
    const int chosen = fa_splitkv_num_splits(B, H, Nq, Nk, d);
    if (chosen < 0)
        return chosen;
    int splits = num_splits == 0 ? chosen : num_splits;
    const int n_kv = (Nk + 127) / 128;
    if (splits > n_kv)
        splits = n_kv;

    // Malformed pointers and sizes the kernels cannot index are reported as
    // fa_attention_fwd_splitkv reports them, before the scratch size is
    // looked at: a call that is both malformed and too big for the array
    // gets the same answer from both functions.
    // (The checks run in fa_attention_fwd_splitkv's order.)
    const int64_t total_q = int64_t(B) * Nq, total_k = int64_t(B) * Nk;
    const int64_t index_limit = (int64_t(1) << 31) - 512;
    if (total_k > index_limit || int64_t(Nk) > index_limit)
        return FA_ERR_TOO_LARGE;
    if (!Q || !K || !V || !O || !lse)
        return FA_ERR_NULL_POINTER;
    const auto aligned = [](const void *p, uintptr_t a) {
        return (reinterpret_cast<uintptr_t>(p) % a) == 0;
    };
    if (!aligned(Q, 16) || !aligned(K, 16) || !aligned(V, 16) || !aligned(O, 16) ||
        !aligned(lse, 4))
        return FA_ERR_MISALIGNED;
    if (total_q > index_limit || total_q * int64_t(H) * int64_t(d) > (int64_t(1) << 56))
        return FA_ERR_TOO_LARGE;

    float *O_accum = nullptr, *lse_accum = nullptr;
    if (splits > 1) {
        // splits * (B * Nq * H) * (d + 1) floats must fit in the array; checked
        // in steps so that no product overflows
        const int64_t cap = int64_t(FA_NOALLOC_SCRATCH_BYTES / sizeof(float));
        const int64_t rows = int64_t(B) * Nq;
        if (rows > cap / H)
            return FA_ERR_SCRATCH_LIMIT;
        const int64_t rows_h = rows * H;
        if (rows_h * (d + 1) > cap / splits)
            return FA_ERR_SCRATCH_LIMIT;
        float *base = nullptr;
        const int rc = fa::scratch_on_current_device(&base);
        if (rc != FA_OK)
            return rc;
        // O_accum [splits, B, Nq, H, d], then lse_accum [splits, B, H, Nq]; the
        // first holds a multiple of 64 floats, so the second stays 256-byte aligned
        O_accum = base;
        lse_accum = base + int64_t(splits) * rows_h * d;
    }
    return fa_attention_fwd_splitkv(Q, K, V, O, lse, B, H, Nq, Nk, d, scale, causal, splits,
                                    O_accum, lse_accum);
}
