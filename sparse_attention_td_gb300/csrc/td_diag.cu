// td_diag.cu -- small kernels around the decode step: KV append and the
// overlap of index sets.
//
// KV append: a decode step appends the new token's K and V rows to the cache
// before attending (the growing KV cache of the decode phase, TidalDecode
// review §二).  One launch writes the rows of up to 32 layers.
//
// Overlap of two top-k sets per (batch row, KV head): the quantity the
// TidalDecode review's token-selection sensitivity analysis plots (§三,
// Figure 4(a): the most attended tokens of consecutive layers overlap
// heavily, which is what lets a set chosen in one layer serve the next).
// Both rows are ascending with -1 padding at the end; read with -1 as +inf
// they stay sorted, so each entry of A is looked up in B by binary search.
#include <cuda_runtime.h>
#include <stdint.h>

#include "td_internal.h"

namespace td {
namespace {

constexpr int kOverlapThreads = 256;

__device__ __forceinline__ uint32_t sort_key(int32_t x)
{
    return x < 0 ? 0xffffffffu : (uint32_t)x;  // padding sorts last
}

__global__ void __launch_bounds__(kOverlapThreads)
overlap_kernel(const int32_t *a, const int32_t *b, int top_k, int32_t *counts)
{
    __shared__ unsigned sm_count;
    const size_t row = blockIdx.x;
    const int32_t *ra = a + row * (size_t)top_k;
    const int32_t *rb = b + row * (size_t)top_k;
    if (threadIdx.x == 0)
        sm_count = 0u;
    __syncthreads();
    unsigned mine = 0;
    for (int j = threadIdx.x; j < top_k; j += kOverlapThreads) {
        const int32_t x = __ldg(ra + j);
        if (x < 0)
            continue;
        // first position in rb whose key is >= x
        int lo = 0, hi = top_k;
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (sort_key(__ldg(rb + mid)) < (uint32_t)x)
                lo = mid + 1;
            else
                hi = mid;
        }
        mine += (lo < top_k && __ldg(rb + lo) == x) ? 1u : 0u;
    }
    for (int off = 16; off >= 1; off >>= 1)
        mine += __shfl_xor_sync(0xffffffffu, mine, off);
    if ((threadIdx.x & 31) == 0 && mine)
        atomicAdd(&sm_count, mine);
    __syncthreads();
    if (threadIdx.x == 0)
        counts[row] = (int32_t)sm_count;
}

// One warp per (batch row, KV head, layer): lanes 0-15 copy the K row, 16-31
// the V row.
__global__ void kv_append_kernel(const AppendBatch layers, const int32_t *seq_lens, int Hkv,
                                 int Nmax)
{
    const int g = blockIdx.x, b = blockIdx.y, l = blockIdx.z, lane = threadIdx.x;
    const int n = seq_lens[b];
    if (n < 1 || n > Nmax)
        return;  // nothing to append (or a length the attention kernels flag)
    const size_t bg = (size_t)b * Hkv + g;
    const int c = lane & 15;
    const uint16_t *src = (lane < 16 ? layers.k_new[l] : layers.v_new[l]) + bg * 128 + c * 8;
    uint16_t *dst = (lane < 16 ? layers.k[l] : layers.v[l]) + (bg * (size_t)Nmax + (n - 1)) * 128 + c * 8;
    *reinterpret_cast<uint4 *>(dst) = *reinterpret_cast<const uint4 *>(src);
}

}  // namespace

cudaError_t launch_index_overlap(const int32_t *a, const int32_t *b, int rows, int top_k,
                                 int32_t *counts, cudaStream_t stream)
{
    if (rows <= 0)
        return cudaSuccess;
    overlap_kernel<<<rows, kOverlapThreads, 0, stream>>>(a, b, top_k, counts);
    return cudaGetLastError();
}

cudaError_t launch_kv_append(const AppendBatch &layers, int num_layers, const int32_t *seq_lens,
                             int batch, int Hkv, int Nmax, cudaStream_t stream)
{
    if (batch <= 0 || Hkv <= 0 || num_layers <= 0)
        return cudaSuccess;
    if (num_layers > kAppendLayers)
        return cudaErrorInvalidValue;
    kv_append_kernel<<<dim3((unsigned)Hkv, (unsigned)batch, (unsigned)num_layers), 32, 0, stream>>>(
        layers, seq_lens, Hkv, Nmax);
    return cudaGetLastError();
}

}  // namespace td
