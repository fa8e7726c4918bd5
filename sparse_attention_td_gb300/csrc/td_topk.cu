// td_topk.cu -- top-k token selection of a TidalDecode selection layer.
//
// "Full Attention + Token Selection -> top-k tokens" (TidalDecode paper
// review, §三 Figure 2; §二 core insight: keep the tokens with the highest
// attention scores).  Per (batch row, KV head) the kernel selects the k
// positions with the largest selection score s[n], n < seq_lens[b] (the
// score the attention kernel emitted: the sum of the group's scaled logits).
// Ties at the k-th score go to the lower position; the result is written in
// ascending position order and padded with -1 when seq_lens[b] < k.
//
// Method: exact radix select on order-preserving 32-bit keys.  Four passes
// of 8-bit digits (most significant first) build a shared-memory histogram
// of the keys that share the prefix found so far and pick the digit holding
// the k-th largest key.  The result is the k-th key T and the number e of
// keys equal to T that belong in the set.  A final pass, in position order,
// keeps every key > T and the first e keys == T, with block-wide ballot
// scans giving each kept position its output slot.
#include <cuda_runtime.h>
#include <stdint.h>

#include "td_internal.h"

namespace td {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kWarps = kTopkThreads / 32;

// Order-preserving key: larger float -> larger unsigned.  -0.0 is mapped to
// +0.0 first so the two tie.
__device__ __forceinline__ uint32_t order_key(float f)
{
    uint32_t u = __float_as_uint(f);
    if (u == 0x80000000u)
        u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Exclusive prefix count of `flag` over the block (thread order), plus the
// block total.  Uses `warp_tot` (kWarps ints) as scratch; contains
// __syncthreads, so every thread must call it.
__device__ __forceinline__ int block_exclusive_count(bool flag, int *warp_tot, int &total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const unsigned bal = __ballot_sync(kFull, flag);
    const int in_warp = __popc(bal & ((1u << lane) - 1u));
    if (lane == 0)
        warp_tot[warp] = __popc(bal);
    __syncthreads();
    int before = 0, all = 0;
    for (int w = 0; w < kWarps; ++w) {
        const int t = warp_tot[w];
        before += (w < warp) ? t : 0;
        all += t;
    }
    __syncthreads();  // warp_tot is reused by the next call
    total = all;
    return before + in_warp;
}

__global__ void __launch_bounds__(kTopkThreads)
topk_kernel(const TopkArgs a)
{
    __shared__ unsigned hist[256];
    __shared__ unsigned sh_digit, sh_krem;
    __shared__ int warp_tot[kWarps];

    const int g = blockIdx.x, b = blockIdx.y, tid = threadIdx.x;
    const size_t bg = (size_t)b * a.Hkv + g;
    const int k = a.top_k;
    int n = a.seq_lens[b];
    if (n < 0 || n > a.Nmax) {
        if (tid == 0 && g == 0)
            atomicOr(a.status, kFlagSeqLenOutOfRange);
        n = n < 0 ? 0 : a.Nmax;
    }
    const float *s = a.scores + bg * (size_t)a.Nmax;
    int32_t *out = a.idx + bg * (size_t)k;

    if (n <= k) {  // every position is kept
        for (int j = tid; j < k; j += kTopkThreads)
            out[j] = j < n ? j : -1;
        return;
    }

    uint32_t prefix = 0u, mask = 0u;
    unsigned krem = (unsigned)k;  // how many of the keys matching `prefix` still belong in the set
    for (int pass = 0; pass < 4; ++pass) {
        const int shift = 24 - 8 * pass;
        for (int i = tid; i < 256; i += kTopkThreads)
            hist[i] = 0u;
        __syncthreads();
        for (int i = tid; i < n; i += kTopkThreads) {
            const uint32_t key = order_key(__ldcg(&s[i]));
            if ((key & mask) == prefix)
                atomicAdd(&hist[(key >> shift) & 255u], 1u);
        }
        __syncthreads();
        if (tid < 32) {
            // lane j owns bins 255-8j down to 248-8j; scan from the top bin down
            const int lane = tid;
            unsigned mine = 0u;
            for (int i = 0; i < 8; ++i)
                mine += hist[255 - 8 * lane - i];
            unsigned incl = mine;
            for (int off = 1; off < 32; off <<= 1) {
                const unsigned v = __shfl_up_sync(kFull, incl, off);
                if (lane >= off)
                    incl += v;
            }
            const unsigned excl = incl - mine;
            if (excl < krem && krem <= incl) {
                unsigned run = excl;
                for (int i = 0; i < 8; ++i) {
                    const int bin = 255 - 8 * lane - i;
                    if (run + hist[bin] >= krem) {
                        sh_digit = (unsigned)bin;
                        sh_krem = krem - run;
                        break;
                    }
                    run += hist[bin];
                }
            }
        }
        __syncthreads();
        prefix |= sh_digit << shift;
        mask |= 255u << shift;
        krem = sh_krem;
        __syncthreads();
    }
    // prefix is now the k-th largest key T; krem keys equal to T are kept.
    const uint32_t T = prefix;
    const int need_eq = (int)krem;
    int out_base = 0, eq_base = 0;
    for (int tile = 0; tile < n; tile += kTopkThreads) {
        const int i = tile + tid;
        uint32_t key = 0u;
        if (i < n)
            key = order_key(__ldcg(&s[i]));
        const bool gt = i < n && key > T;
        const bool eq = i < n && key == T;
        int eq_total = 0, take_total = 0;
        const int eq_rank = eq_base + block_exclusive_count(eq, warp_tot, eq_total);
        const bool take = gt || (eq && eq_rank < need_eq);
        const int slot = out_base + block_exclusive_count(take, warp_tot, take_total);
        if (take && slot < k)  // exactly k are taken; the bound only guards memory
            out[slot] = i;
        out_base += take_total;
        eq_base += eq_total;
    }
}

}  // namespace

cudaError_t launch_topk(const TopkArgs &a, int batch, cudaStream_t stream)
{
    dim3 grid((unsigned)a.Hkv, (unsigned)batch);
    topk_kernel<<<grid, kTopkThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace td
