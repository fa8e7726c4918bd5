// td_diag.cu -- small kernels around the decode step: KV append, the
// overlap of index sets, and a read probe for measurement.
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

// Measurement aid: the K/V reads of one attention launch and nothing else.
// Same grid, split plan, index staging and 16-byte row loads (4 tokens of K
// and V in flight per thread) as the register-streamed attention kernel; the
// data only feed an XOR, one word of which each CTA stores.
constexpr int kProbeThreads = 256;
constexpr int kProbeTok = 4;

__global__ void __launch_bounds__(kProbeThreads)
probe_reads_kernel(const ProbeArgs a)
{
    __shared__ int sm_rows[kMaxSparseChunk];
    const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int half = lane >> 4, c = lane & 15;
    int n_b = a.seq_lens[b];
    n_b = n_b < 0 ? 0 : (n_b > a.Nmax ? a.Nmax : n_b);
    const bool sparse = a.idx != nullptr;
    const int n_total = sparse ? a.top_k : n_b;
    const int t0 = split * a.chunk;
    const int t1 = min(t0 + a.chunk, n_total);
    if (t0 >= t1)
        return;
    const size_t bg = (size_t)b * a.Hkv + g;
    const uint16_t *kb = a.k + bg * (size_t)a.Nmax * 128 + c * 8;
    const uint16_t *vb = a.v + bg * (size_t)a.Nmax * 128 + c * 8;
    if (sparse) {
        const int32_t *ip = a.idx + bg * (size_t)a.top_k;
        for (int j = tid; j < t1 - t0; j += kProbeThreads) {
            const int r = ip[t0 + j];
            sm_rows[j] = (r >= 0 && r < n_b) ? r : -1;
        }
        __syncthreads();
    }
    unsigned acc = 0;
    for (int base = t0; base < t1; base += kProbeThreads / 16 * kProbeTok) {
        const int tb = base + (warp * 2 + half) * kProbeTok;
        uint4 kr[kProbeTok], vr[kProbeTok];
#pragma unroll
        for (int u = 0; u < kProbeTok; ++u) {
            const int t = tb + u;
            const int row = t < t1 ? (sparse ? sm_rows[t - t0] : t) : -1;
            kr[u] = make_uint4(0u, 0u, 0u, 0u);
            vr[u] = kr[u];
            if (row >= 0) {
                asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                             : "=r"(kr[u].x), "=r"(kr[u].y), "=r"(kr[u].z), "=r"(kr[u].w)
                             : "l"(kb + (size_t)row * 128));
                asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                             : "=r"(vr[u].x), "=r"(vr[u].y), "=r"(vr[u].z), "=r"(vr[u].w)
                             : "l"(vb + (size_t)row * 128));
            }
        }
        // every load of the round is issued before any of them is used
#pragma unroll
        for (int u = 0; u < kProbeTok; ++u)
            asm volatile("" : "+r"(kr[u].x), "+r"(kr[u].y), "+r"(kr[u].z), "+r"(kr[u].w),
                         "+r"(vr[u].x), "+r"(vr[u].y), "+r"(vr[u].z), "+r"(vr[u].w));
#pragma unroll
        for (int u = 0; u < kProbeTok; ++u)
            acc ^= kr[u].x ^ kr[u].y ^ kr[u].z ^ kr[u].w ^ vr[u].x ^ vr[u].y ^ vr[u].z ^ vr[u].w;
    }
    for (int off = 16; off >= 1; off >>= 1)
        acc ^= __shfl_xor_sync(0xffffffffu, acc, off);
    if (lane == 0)
        atomicXor(a.sink + (bg * (size_t)gridDim.x + split) % a.sink_words, acc);
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

cudaError_t launch_probe_reads(const ProbeArgs &a, int batch, cudaStream_t stream)
{
    if (batch <= 0 || a.Hkv <= 0 || a.nsplit <= 0)
        return cudaSuccess;
    probe_reads_kernel<<<dim3((unsigned)a.nsplit, (unsigned)a.Hkv, (unsigned)batch), kProbeThreads, 0,
                         stream>>>(a);
    return cudaGetLastError();
}

}  // namespace td
