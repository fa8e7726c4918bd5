// td_attn_mma.cu -- grouped-query attention on the tensor cores (G = 4, 8).
//
// The same layer math as td_attn.cu (TidalDecode paper review, §三:
// A = q K^T / sqrt(d), H = softmax(A) V, split over the token axis, full or
// over the persisted positions), with both contractions over a KV head's G
// query heads done by mma.sync m16n8k16 (bf16 inputs, fp32 accumulation):
//   S[token][head] = K Q^T   (M = tokens, N = heads padded to 8, K = dims)
//   O[dim][head]  += V^T P^T (M = dims,   N = heads,              K = tokens)
// Three kernels, the same arithmetic, different tiling:
//   * attention_mma_kernel: a warp takes 8 tokens per round (MMA rows 8..15
//     of S and tokens 8..15 of the P V k-step stay zero), a CTA of 8 warps
//     64 tokens; 2 CTAs per SM.
//   * attention_mma_ring_kernel: the same 8-token rounds for sparse layers,
//     gathered into a ring of two shared-memory stages by cp.async and read
//     back by ldmatrix, one round in flight ahead of the one computed.
//     Default for sparse layers.
//   * attention_mma16_kernel: a warp takes 16 tokens per round (rows r and
//     r + 8 of S are two tokens, the P V k-step takes all 16), a CTA of 4
//     warps 64 tokens; half the MMAs and shuffles per token, 3 CTAs per SM.
//     Default for full and full+select layers.
// Measured on GB300: the 16-token kernel takes 2-6% off full and full+select
// layers, but is slower on sparse layers whose CTAs are short and
// latency-bound.  The splits of each merge as in the CUDA-core kernels.
//
// In the first and last kernels fragments come straight from global memory
// (the ring kernel's layout is described with it).  The dot product does not care
// in which order the 128 dims are summed, so k-step j of the S product maps
// MMA column pairs {2c, 2c+1} / {2c+8, 2c+9} of lane quad position c to dims
// 16j + 4c + {0,1} / {2,3}: a lane reads 8 bytes of its token's K row (and of
// its head's q row) per k-step, and a quad reads 32 contiguous bytes -- whole
// sectors.  For O, MMA rows r / r+8 of m-tile i are the two dims of word i of
// lane row r's V slice: dims 8r .. 8r+7 (tiles 0-3) and 64+8r .. 64+8r+7
// (tiles 4-7), so 8 lanes read 128 contiguous bytes per load; O is written
// back in natural order.
//
// P goes into the tensor cores as bf16, so it is split into three bf16 terms
// (p = p1 + p2 + p3 to about 2^-24 relative) and O accumulates all three:
// the fp32 result keeps fp32 accuracy.  K, V and q are bf16 already, so the
// S product is exact up to fp32 summation order.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math_constants.h>
#include <stdint.h>

#include "td_attn_common.cuh"
#include "td_internal.h"

namespace td {
namespace {

// Not volatile: the compiler may interleave independent MMAs (different
// accumulators) with each other and with the loads, instead of issuing each
// right behind the one it depends on.
__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1)
{
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// 16-byte read-only load, no L1 allocation (8 lanes cover 128 contiguous bytes).
__device__ __forceinline__ uint4 ldg16(const uint16_t *p)
{
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// 8-byte read-only load (a quad covers whole 32-byte sectors per instruction).
__device__ __forceinline__ uint2 ldg8(const uint16_t *p)
{
    uint2 r;
    asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0, %1}, [%2];"
                 : "=r"(r.x), "=r"(r.y)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ uint32_t word2(const uint4 (&v)[2], int w)
{
    const uint4 &x = v[w >> 2];
    return (w & 3) == 0 ? x.x : (w & 3) == 1 ? x.y : (w & 3) == 2 ? x.z : x.w;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel)
{
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

template <int G, bool SPARSE, bool SELECT>
__global__ void __launch_bounds__(kAttnThreads, 2)
attention_mma_kernel(const AttnArgs a)
{
    static_assert(G == 4 || G == 8, "heads of a group are the MMA's N = 8 columns");
    __shared__ float sm_m[kAttnWarps][G];
    __shared__ float sm_l[kAttnWarps][G];
    __shared__ float sm_w[kAttnWarps][G];
    __shared__ __align__(16) float sm_o[kAttnWarps][G][kHeadDim];
    __shared__ float sm_M[G];
    __shared__ float sm_L[G];
    __shared__ int sm_rows[SPARSE ? kMaxSparseChunk : 1];
    __shared__ int sm_last;
    __shared__ unsigned sm_hist[SELECT ? kSelectBins : 1];

    const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int r = lane >> 2, c = lane & 3;  // MMA fragment row group / quad position

    int n_b = a.seq_lens[b];
    if (n_b < 0 || n_b > a.Nmax) {
        if (tid == 0)
            atomicOr(a.status, kFlagSeqLenOutOfRange);
        n_b = n_b < 0 ? 0 : a.Nmax;
    }
    const int n_total = SPARSE ? a.top_k : n_b;
    const int nsplit_b = n_total > 0 ? (n_total + a.chunk - 1) / a.chunk : 1;
    if (split >= nsplit_b)
        return;
    const int t0 = split * a.chunk;
    const int t1 = min(t0 + a.chunk, n_total);
    const size_t bg = (size_t)b * a.Hkv + g;
    const uint16_t *kbase = a.k + bg * (size_t)a.Nmax * kHeadDim;
    const uint16_t *vbase = a.v + bg * (size_t)a.Nmax * kHeadDim;

    if constexpr (SELECT) {
        for (int i = tid; i < kSelectBins; i += kAttnThreads)
            sm_hist[i] = 0u;
        __syncthreads();
    }
    if constexpr (SPARSE) {
        if (a.idx_dep)
            pdl_wait();
        const int32_t *ip = a.idx + bg * (size_t)a.top_k;
        for (int j = tid; j < t1 - t0; j += kAttnThreads) {
            int rr = ip[t0 + j];
            if (rr < -1 || rr >= n_b) {
                atomicOr(a.status, kFlagIndexOutOfRange);
                rr = -1;
            }
            sm_rows[j] = rr;
        }
        __syncthreads();
    }
    auto row_of = [&](int t) { return t < t1 ? (SPARSE ? sm_rows[t - t0] : t) : -1; };

    // This warp's 8 tokens of the round at `base`: K of token r (dims
    // 16j + 4c .. +3 for k-step j) and V of tokens 2c, 2c+1 (dims 8r..8r+7 and
    // 64+8r..64+8r+7).
    auto load = [&](int base, uint2 (&kq)[8], uint4 (&v0)[2], uint4 (&v1)[2]) {
        const int tw = base + warp * 8;
        const int rk = row_of(tw + r);
        const int r0 = row_of(tw + 2 * c), r1 = row_of(tw + 2 * c + 1);
#pragma unroll
        for (int j = 0; j < 8; ++j)
            kq[j] = rk >= 0 ? ldg8(kbase + (size_t)rk * kHeadDim + 16 * j + 4 * c)
                            : make_uint2(0u, 0u);
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            v0[i] = r0 >= 0 ? ldg16(vbase + (size_t)r0 * kHeadDim + 64 * i + 8 * r)
                            : make_uint4(0u, 0u, 0u, 0u);
            v1[i] = r1 >= 0 ? ldg16(vbase + (size_t)r1 * kHeadDim + 64 * i + 8 * r)
                            : make_uint4(0u, 0u, 0u, 0u);
        }
    };
    uint2 kq0[8];
    uint4 va0[2], vb0[2];
    load(t0, kq0, va0, vb0);  // the cache is never written by a kernel of the step
    // full layers: rounds 1 .. prefetch go to L2 now, later rounds `prefetch`
    // ahead of use (measured on GB300: no gain for gathered rows)
    const int pf = SPARSE ? 0 : a.prefetch;
    for (int d = 1; d <= pf; ++d)
        prefetch_round_l2(kbase, vbase, t0 + d * kTokPerRound + warp * 8, lane, row_of);
    pdl_wait();

    // q of head r (heads >= G are zero columns): dims 16j + 4c .. +3.
    uint2 qf[8];
#pragma unroll
    for (int j = 0; j < 8; ++j)
        qf[j] = r < G ? *reinterpret_cast<const uint2 *>(
                            a.q + ((size_t)b * a.Hq + (size_t)g * G + r) * kHeadDim + 16 * j + 4 * c)
                      : make_uint2(0u, 0u);

    const float c2 = a.scale * kLog2e;
    float m[2] = {-CUDART_INF_F, -CUDART_INF_F};  // heads 2c, 2c+1 (replicated over r)
    float l[2] = {0.0f, 0.0f};
    // m-tile i holds dims vdim(i) (0, 1: heads 2c, 2c+1) and vdim(i) + 1 (2, 3),
    // vdim(i) = (i < 4 ? 8r : 64 + 8r) + 2 (i % 4)
    float o[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j)
            o[i][j] = 0.0f;

    auto round = [&](int base, const uint2 (&kq)[8], const uint4 (&v0)[2], const uint4 (&v1)[2]) {
        const int tw = base + warp * 8;
        // two accumulators (even / odd k-steps): two chains of 4 dependent MMAs
        float s[4] = {0.0f, 0.0f, 0.0f, 0.0f}, s_odd[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
        for (int j = 0; j < 8; j += 2) {
            mma_bf16(s, kq[j].x, 0u, kq[j].y, 0u, qf[j].x, qf[j].y);
            mma_bf16(s_odd, kq[j + 1].x, 0u, kq[j + 1].y, 0u, qf[j + 1].x, qf[j + 1].y);
        }
#pragma unroll
        for (int e = 0; e < 4; ++e)
            s[e] += s_odd[e];
        const bool ok = row_of(tw + r) >= 0;

        if constexpr (SELECT) {
            // selection score of token tw + r: the group's summed scaled logits
            float sc = (2 * c < G ? s[0] * a.scale : 0.0f) + (2 * c + 1 < G ? s[1] * a.scale : 0.0f);
            sc += __shfl_xor_sync(kFull, sc, 1);
            sc += __shfl_xor_sync(kFull, sc, 2);
            if (c == 0 && tw + r < t1) {
                a.scores[bg * (size_t)a.Nmax + tw + r] = sc;
                atomicAdd(&sm_hist[order_key(sc) >> (32 - kSelectBits)], 1u);
            }
        }

        // online softmax of heads 2c, 2c+1 over the warp's 8 tokens
        float p[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const bool head = 2 * c + e < G;
            const float x = (ok && head) ? s[e] * c2 : -CUDART_INF_F;
            float mx = x;
            mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 4));
            mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 8));
            mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 16));
            const float m_new = fmaxf(m[e], mx);
            float alpha = 1.0f;
            p[e] = 0.0f;
            if (m_new != -CUDART_INF_F) {  // uniform over the 8 lanes of this head
                alpha = safe_exp2_diff(m[e], m_new);
                p[e] = (x == -CUDART_INF_F) ? 0.0f : exp2f(x - m_new);
            }
            float ps = p[e];
            ps += __shfl_xor_sync(kFull, ps, 4);
            ps += __shfl_xor_sync(kFull, ps, 8);
            ps += __shfl_xor_sync(kFull, ps, 16);
            if (m_new != -CUDART_INF_F) {
                l[e] = l[e] * alpha + ps;
                m[e] = m_new;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    o[i][e] *= alpha;
                    o[i][e + 2] *= alpha;
                }
            }
        }

        // P^T fragment: P[token 2c][head r], P[token 2c+1][head r], held by
        // lanes (row 2c / 2c+1, quad r / 2) in register r & 1
        const int src0 = 8 * c + (r >> 1), src1 = 8 * c + 4 + (r >> 1);
        const float a0p = __shfl_sync(kFull, p[0], src0), a1p = __shfl_sync(kFull, p[1], src0);
        const float b0p = __shfl_sync(kFull, p[0], src1), b1p = __shfl_sync(kFull, p[1], src1);
        float pt0 = (r & 1) ? a1p : a0p;
        float pt1 = (r & 1) ? b1p : b0p;
        uint32_t pb[3];
#pragma unroll
        for (int k = 0; k < 3; ++k) {  // p = p1 + p2 + p3 in bf16
            const __nv_bfloat16 h0 = __float2bfloat16_rn(pt0), h1 = __float2bfloat16_rn(pt1);
            pb[k] = (uint32_t)__bfloat16_as_ushort(h0) | ((uint32_t)__bfloat16_as_ushort(h1) << 16);
            pt0 -= __bfloat162float(h0);
            pt1 -= __bfloat162float(h1);
        }
        // O += V^T P^T, m-tiles of 16 dims; the three terms of P in the
        // outer loop, so that consecutive MMAs go to different tiles
        uint32_t lo[8], hi[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t w0 = word2(v0, i), w1 = word2(v1, i);
            lo[i] = prmt(w0, w1, 0x5410u);  // dim vdim(i) of tokens 2c, 2c+1
            hi[i] = prmt(w0, w1, 0x7632u);  // dim vdim(i) + 1
        }
#pragma unroll
        for (int k = 0; k < 3; ++k)
#pragma unroll
            for (int i = 0; i < 8; ++i)
                mma_bf16(o[i], lo[i], hi[i], 0u, 0u, pb[k], 0u);
    };

    if (t0 < t1)
        round(t0, kq0, va0, vb0);
    for (int base = t0 + kTokPerRound; base < t1; base += kTokPerRound) {
        uint2 kq[8];
        uint4 va[2], vb[2];
        if (pf > 0)
            prefetch_round_l2(kbase, vbase, base + pf * kTokPerRound + warp * 8, lane, row_of);
        load(base, kq, va, vb);
        round(base, kq, va, vb);
    }

    pdl_launch_dependents();

    // this warp's partial into shared memory (dims back in natural order)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        const int h = 2 * c + e;
        if (h < G) {
            if (r == 0) {
                sm_m[warp][h] = m[e];
                sm_l[warp][h] = l[e];
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int d = (i < 4 ? 8 * r : 64 + 8 * r) + 2 * (i & 3);
                sm_o[warp][h][d] = o[i][e];
                sm_o[warp][h][d + 1] = o[i][e + 2];
            }
        }
    }
    __syncthreads();
    if constexpr (SELECT) {
        unsigned *gh = a.hist + bg * kSelectBins;
        for (int i = tid; i < kSelectBins; i += kAttnThreads)
            if (sm_hist[i])
                atomicAdd(&gh[i], sm_hist[i]);
    }
    if (tid < G) {
        const int h = tid;
        float M = -CUDART_INF_F;
        for (int w = 0; w < kAttnWarps; ++w)
            M = fmaxf(M, sm_m[w][h]);
        float L = 0.0f;
        for (int w = 0; w < kAttnWarps; ++w) {
            const float wt = safe_exp2_diff(sm_m[w][h], M);
            sm_w[w][h] = wt;
            L += sm_l[w][h] * wt;
        }
        sm_M[h] = M;
        sm_L[h] = L;
    }
    __syncthreads();
    const size_t out_row0 = (size_t)b * a.Hq + (size_t)g * G;
    finish_splits<G>(a, sm_o, sm_w, sm_M, sm_L, &sm_last, bg, split, nsplit_b, out_row0);
}

// Sparse layers through a ring of shared-memory stages: a stage holds one
// CTA round of gathered rows (64 K rows and their 64 V rows, 32 KB) copied by
// cp.async, 16 bytes a lane and copy; each warp gathers the 8 rows it
// computes, so warps wait only for their own copies (no block barrier in the
// loop).  kRingStages stages, so kRingStages - 1 rounds are in flight while
// one is computed, and the first of them are requested before the wait for
// the previous kernel.  Padding and positions
// past the split are zero-filled (their logits are masked; V must stay
// finite).  The 16-byte chunks of each stored row are XOR-swizzled by the row
// (chunk q of row t at q ^ (t & 7)), so the 8 row addresses of one ldmatrix
// fall in 8 different bank groups.  Fragments take the standard m16n8k16
// layout, straight from ldmatrix:
//   S = K q^T: A = K of the warp's 8 tokens (rows 8..15 zero), k-step j =
//     dims 16j .. 16j + 15; B = q^T, dims 16j + 2c, +1 and 16j + 8 + 2c, +1
//     of head r (loaded once from global);
//   O += V^T P^T: A = V^T by ldmatrix.trans, rows r / r + 8 of m-tile t =
//     dims 16t + r / 16t + 8 + r, k = the warp's 8 tokens (8..15 zero);
//     B = P^T as in attention_mma_kernel.
// The warps' partial outputs reuse the ring once the last round is done.
// Measured on GB300 (graph steps, outputs bitwise equal): two stages against
// three take 32K 730.8 -> 688.2 us, serving batch k = 1024 1751.7 -> 1697.1
// us, and at k = 256 the ring beats the 8-token kernel, 1279.8 -> 1237.5 us
// (three stages: 1314.5 us).
constexpr int kRingStages = 2;
constexpr int kRingRowBytes = kHeadDim * 2;                          // 256
constexpr int kRingStageBytes = 2 * kTokPerRound * kRingRowBytes;    // K block + V block
constexpr int kRingSmemBytes = kRingStages * kRingStageBytes;        // 64 KB

__device__ __forceinline__ uint32_t shared_addr(const void *p)
{
    return (uint32_t)__cvta_generic_to_shared(p);
}

// 16-byte global -> shared copy through L2 (cp.async.cg); zero-fills the
// destination instead when !valid (src is then not read).
__device__ __forceinline__ void cp_async16_or_zero(uint32_t dst, const void *src, bool valid)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
                 "r"(valid ? 16 : 0)
                 : "memory");
}

__device__ __forceinline__ void cp_async_commit_group()
{
    asm volatile("cp.async.commit_group;" ::: "memory");
}

template <int N>
__device__ __forceinline__ void cp_async_wait_group()
{
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Four 8x8 bf16 matrices from shared memory; lanes 8m .. 8m + 7 give the row
// addresses of matrix m, register m receives its fragment.
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &d0, uint32_t &d1, uint32_t &d2,
                                        uint32_t &d3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(d0), "=r"(d1), "=r"(d2), "=r"(d3)
                 : "r"(addr)
                 : "memory");
}

// The same, each matrix transposed.
__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t &d0, uint32_t &d1,
                                              uint32_t &d2, uint32_t &d3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(d0), "=r"(d1), "=r"(d2), "=r"(d3)
                 : "r"(addr)
                 : "memory");
}

template <int G>
__global__ void __launch_bounds__(kAttnThreads, 2)
attention_mma_ring_kernel(const AttnArgs a)
{
    static_assert(G == 4 || G == 8, "heads of a group are the MMA's N = 8 columns");
    static_assert(kAttnWarps * G * kHeadDim * 4 <= kRingSmemBytes, "sm_o fits in the ring");
    extern __shared__ __align__(128) unsigned char ring[];
    __shared__ float sm_m[kAttnWarps][G];
    __shared__ float sm_l[kAttnWarps][G];
    __shared__ float sm_w[kAttnWarps][G];
    __shared__ float sm_M[G];
    __shared__ float sm_L[G];
    __shared__ int sm_rows[kMaxSparseChunk];
    __shared__ int sm_last;
    float(*sm_o)[G][kHeadDim] = reinterpret_cast<float(*)[G][kHeadDim]>(ring);

    const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int r = lane >> 2, c = lane & 3;  // MMA fragment row group / quad position

    // the length check reports after the index entries are requested
    const int n_raw = a.seq_lens[b];
    const int n_b = n_raw < 0 ? 0 : (n_raw > a.Nmax ? a.Nmax : n_raw);
    const int n_total = a.top_k;
    const int nsplit_b = n_total > 0 ? (n_total + a.chunk - 1) / a.chunk : 1;
    if (split >= nsplit_b)
        return;
    const int t0 = split * a.chunk;
    const int t1 = min(t0 + a.chunk, n_total);
    const size_t bg = (size_t)b * a.Hkv + g;
    const uint16_t *kbase = a.k + bg * (size_t)a.Nmax * kHeadDim;
    const uint16_t *vbase = a.v + bg * (size_t)a.Nmax * kHeadDim;

    if (a.idx_dep)
        pdl_wait();
    stage_index_rows<kAttnThreads>(a.idx + bg * (size_t)a.top_k, t0, t1 - t0, n_b, a.status,
                                   sm_rows, tid);
    if (tid == 0 && n_raw != n_b)
        atomicOr(a.status, kFlagSeqLenOutOfRange);
    __syncthreads();

    // Stage `it` holds the rows of tokens t0 + 64 it ..; each warp copies the
    // 8 rows it computes (stage rows 8 warp ..), one token per step: lanes
    // 0-15 the K row's 16-byte chunks, lanes 16-31 the V row's.
    const int n_it = (t1 - t0 + kTokPerRound - 1) / kTokPerRound;
    const uint32_t ring_s = shared_addr(ring);
    auto issue = [&](int it) {
        const uint32_t st = ring_s + (uint32_t)((it % kRingStages) * kRingStageBytes);
        const int tl = t0 + it * kTokPerRound + warp * 8 + (lane & 7);
        const int pl = tl < t1 ? sm_rows[tl - t0] : -1;
        const int q = lane & 15;
        const uint32_t dst0 = st + (lane < 16 ? 0u : (uint32_t)(kRingStageBytes / 2)) +
                              (uint32_t)(warp * 8 * kRingRowBytes);
        const uint16_t *src0 = (lane < 16 ? kbase : vbase) + q * 8;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int p = __shfl_sync(kFull, pl, j);
            cp_async16_or_zero(dst0 + (uint32_t)(j * kRingRowBytes + ((q ^ j) << 4)),
                               src0 + (size_t)(p >= 0 ? p : 0) * kHeadDim, p >= 0);
        }
    };
    // the cache is never written by a kernel of the step
    for (int st = 0; st < kRingStages - 1; ++st) {
        if (st < n_it)
            issue(st);
        cp_async_commit_group();
    }
    pdl_wait();

    // q^T fragments of head r (heads >= G are zero columns)
    uint32_t qb0[8], qb1[8];
    {
        const uint16_t *qrow = a.q + ((size_t)b * a.Hq + (size_t)g * G + r) * kHeadDim;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            qb0[j] = r < G ? *reinterpret_cast<const uint32_t *>(qrow + 16 * j + 2 * c) : 0u;
            qb1[j] = r < G ? *reinterpret_cast<const uint32_t *>(qrow + 16 * j + 8 + 2 * c) : 0u;
        }
    }

    const float c2 = a.scale * kLog2e;
    float m[2] = {-CUDART_INF_F, -CUDART_INF_F};  // heads 2c, 2c+1 (replicated over r)
    float l[2] = {0.0f, 0.0f};
    // m-tile t: o[t][0, 1] = O[dim 16t + r][heads 2c, 2c+1], o[t][2, 3] = dim 16t + 8 + r
    float o[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j)
            o[i][j] = 0.0f;

    const int lrow = warp * 8 + (lane & 7);  // stage row whose address this lane gives ldmatrix
    const int lmat = lane >> 3;              // the matrix of the x4 it belongs to
    for (int it = 0; it < n_it; ++it) {
        if (a.early_trigger > 0 && it == max(n_it - a.early_trigger, 0))
            pdl_launch_dependents();
        if (it + kRingStages - 1 < n_it)
            issue(it + kRingStages - 1);  // into the slice this warp finished last round
        cp_async_commit_group();
        cp_async_wait_group<kRingStages - 1>();  // this lane's copies of stage `it` landed
        __syncwarp();                            // ... and the other lanes' of this warp
        const uint32_t kst = ring_s + (uint32_t)((it % kRingStages) * kRingStageBytes);
        const uint32_t vst = kst + kRingStageBytes / 2;
        const uint32_t lrow_off = (uint32_t)(lrow * kRingRowBytes);
        const int tw = t0 + it * kTokPerRound + warp * 8;  // this warp's 8 tokens

        // S = K q^T: ldmatrix x4 jj gives k-steps 2jj and 2jj + 1 (dim chunks 4jj .. 4jj + 3)
        float s[4] = {0.0f, 0.0f, 0.0f, 0.0f}, s_odd[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
            const int q = 4 * jj + lmat;
            uint32_t k0, k1, k2, k3;
            ldsm_x4(kst + lrow_off + (uint32_t)((q ^ (lrow & 7)) << 4), k0, k1, k2, k3);
            mma_bf16(s, k0, 0u, k1, 0u, qb0[2 * jj], qb1[2 * jj]);
            mma_bf16(s_odd, k2, 0u, k3, 0u, qb0[2 * jj + 1], qb1[2 * jj + 1]);
        }
#pragma unroll
        for (int e = 0; e < 4; ++e)
            s[e] += s_odd[e];
        const bool ok = tw + r < t1 && sm_rows[tw + r - t0] >= 0;

        // online softmax of heads 2c, 2c+1 over the warp's 8 tokens
        float p[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const bool head = 2 * c + e < G;
            const float x = (ok && head) ? s[e] * c2 : -CUDART_INF_F;
            float mx = x;
            mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 4));
            mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 8));
            mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 16));
            const float m_new = fmaxf(m[e], mx);
            float alpha = 1.0f;
            p[e] = 0.0f;
            if (m_new != -CUDART_INF_F) {  // uniform over the 8 lanes of this head
                alpha = safe_exp2_diff(m[e], m_new);
                p[e] = (x == -CUDART_INF_F) ? 0.0f : exp2f(x - m_new);
            }
            float ps = p[e];
            ps += __shfl_xor_sync(kFull, ps, 4);
            ps += __shfl_xor_sync(kFull, ps, 8);
            ps += __shfl_xor_sync(kFull, ps, 16);
            if (m_new != -CUDART_INF_F) {
                l[e] = l[e] * alpha + ps;
                m[e] = m_new;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    o[i][e] *= alpha;
                    o[i][e + 2] *= alpha;
                }
            }
        }

        // P^T fragment: P[token 2c][head r], P[token 2c+1][head r], held by
        // lanes (row 2c / 2c+1, quad r / 2) in register r & 1
        const int src0 = 8 * c + (r >> 1), src1 = 8 * c + 4 + (r >> 1);
        const float a0p = __shfl_sync(kFull, p[0], src0), a1p = __shfl_sync(kFull, p[1], src0);
        const float b0p = __shfl_sync(kFull, p[0], src1), b1p = __shfl_sync(kFull, p[1], src1);
        float pt0 = (r & 1) ? a1p : a0p;
        float pt1 = (r & 1) ? b1p : b0p;
        uint32_t pb[3];
#pragma unroll
        for (int k = 0; k < 3; ++k) {  // p = p1 + p2 + p3 in bf16
            const __nv_bfloat16 h0 = __float2bfloat16_rn(pt0), h1 = __float2bfloat16_rn(pt1);
            pb[k] = (uint32_t)__bfloat16_as_ushort(h0) | ((uint32_t)__bfloat16_as_ushort(h1) << 16);
            pt0 -= __bfloat162float(h0);
            pt1 -= __bfloat162float(h1);
        }
        // O += V^T P^T: ldmatrix.trans x4 tt gives rows r and r + 8 of m-tiles
        // 2tt and 2tt + 1 (dim chunks 4tt .. 4tt + 3)
        uint32_t va[8], vb[8];
#pragma unroll
        for (int tt = 0; tt < 4; ++tt) {
            const int q = 4 * tt + lmat;
            ldsm_x4_trans(vst + lrow_off + (uint32_t)((q ^ (lrow & 7)) << 4), va[2 * tt],
                          vb[2 * tt], va[2 * tt + 1], vb[2 * tt + 1]);
        }
#pragma unroll
        for (int k = 0; k < 3; ++k)
#pragma unroll
            for (int i = 0; i < 8; ++i)
                mma_bf16(o[i], va[i], vb[i], 0u, 0u, pb[k], 0u);
        __syncwarp();  // every lane is done with this slice before it is refilled
    }

    pdl_launch_dependents();
    __syncthreads();  // every warp is done with the ring, which sm_o reuses

    // this warp's partial into shared memory
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        const int h = 2 * c + e;
        if (h < G) {
            if (r == 0) {
                sm_m[warp][h] = m[e];
                sm_l[warp][h] = l[e];
            }
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                sm_o[warp][h][16 * t + r] = o[t][e];
                sm_o[warp][h][16 * t + 8 + r] = o[t][e + 2];
            }
        }
    }
    __syncthreads();
    if (tid < G) {
        const int h = tid;
        float M = -CUDART_INF_F;
        for (int w = 0; w < kAttnWarps; ++w)
            M = fmaxf(M, sm_m[w][h]);
        float L = 0.0f;
        for (int w = 0; w < kAttnWarps; ++w) {
            const float wt = safe_exp2_diff(sm_m[w][h], M);
            sm_w[w][h] = wt;
            L += sm_l[w][h] * wt;
        }
        sm_M[h] = M;
        sm_L[h] = L;
    }
    __syncthreads();
    const size_t out_row0 = (size_t)b * a.Hq + (size_t)g * G;
    finish_splits<G>(a, sm_o, sm_w, sm_M, sm_L, &sm_last, bg, split, nsplit_b, out_row0);
}

// 16 tokens per warp per round, CTAs of 4 warps (kTokPerRound tokens a CTA
// round).  Fragment maps as in attention_mma_kernel, with the MMAs' second
// row group filled: K of tokens r and r + 8 (A rows r, r + 8 of S); V of
// tokens 2c, 2c+1, 2c+8, 2c+9 (the P V k-step's 16 tokens); P of the same
// four tokens per head.
// DB = false: one round in flight per warp, at most 168 registers (3 CTAs per
// SM).  DB = true: two register buffers, the next round's rows are requested
// before this round's arithmetic (twice the bytes in flight per warp), at
// most 255 registers (2 CTAs per SM).
constexpr int kMma16Warps = kTokPerRound / 16;
constexpr int kMma16Threads = kMma16Warps * 32;

// SK (sparse only): stream-K partition of the launch.  The grid is 1D; the
// layer's B * Hkv * R rounds (R = rounds of 64 index entries per (batch row,
// KV head)) are split evenly over the CTAs, so every CTA gets the same number
// of rounds and a CTA's range may cover the end of one (batch row, KV head)
// and the start of the next.  It publishes one partial per (batch row, KV
// head) it touched; the split merge counts, per (batch row, KV head), the CTAs
// whose ranges meet it.  Without SK: one CTA per (split, KV head, batch row).
template <int G, bool SPARSE, bool SELECT, bool DB, bool SK = false>
__global__ void __launch_bounds__(kMma16Threads, DB ? 2 : 3)
attention_mma16_kernel(const AttnArgs a)
{
    static_assert(G == 4 || G == 8, "heads of a group are the MMA's N = 8 columns");
    static_assert(!SK || SPARSE, "the stream-K partition serves sparse layers");
    constexpr int NW = kMma16Warps, NT = kMma16Threads;
    __shared__ float sm_m[NW][G];
    __shared__ float sm_l[NW][G];
    __shared__ float sm_w[NW][G];
    __shared__ __align__(16) float sm_o[NW][G][kHeadDim];
    __shared__ float sm_M[G];
    __shared__ float sm_L[G];
    __shared__ int sm_rows[SPARSE ? kMaxSparseChunk : 1];
    __shared__ int sm_last;
    __shared__ unsigned sm_hist[SELECT ? kSelectBins : 1];

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int r = lane >> 2, c = lane & 3;  // MMA fragment row group / quad position

    // SK: this CTA's rounds [x, x_end) of the layer's W rounds, R per (batch
    // row, KV head); CTA p covers [floor(p W / P), floor((p + 1) W / P)).
    const long R = SK ? (a.top_k + kTokPerRound - 1) / kTokPerRound : 1;
    const long W = SK ? (long)a.sk_units * R : 1;
    const long P = SK ? gridDim.x : 1;
    long x = SK ? (long)blockIdx.x * W / P : 0;
    const long x_end = SK ? ((long)blockIdx.x + 1) * W / P : 1;
    for (bool first = true; x < x_end; first = false) {
    int split, g, b, t0, t1, nsplit_b;
    if constexpr (SK) {
        // the (batch row, KV head) u of round x, the CTAs meeting it, and this
        // CTA's place among them (the CTA holding round y is
        // floor(((y + 1) P - 1) / W))
        const long u = x / R;
        const long seg_end = min(x_end, (u + 1) * R);
        const long p_first = ((u * R + 1) * P - 1) / W;
        const long p_last = ((u + 1) * R * P - 1) / W;
        split = (int)(blockIdx.x - p_first);
        nsplit_b = (int)(p_last - p_first + 1);
        b = (int)(u / a.Hkv);
        g = (int)(u % a.Hkv);
        t0 = (int)((x - u * R) * kTokPerRound);
        t1 = min((int)((seg_end - u * R) * kTokPerRound), a.top_k);
        x = seg_end;
        if (!first)
            __syncthreads();  // the previous segment is done with shared memory
    } else {
        split = blockIdx.x;
        g = blockIdx.y;
        b = blockIdx.z;
        x = x_end;
    }
    (void)first;

    int n_b = a.seq_lens[b];
    if (n_b < 0 || n_b > a.Nmax) {
        if (tid == 0)
            atomicOr(a.status, kFlagSeqLenOutOfRange);
        n_b = n_b < 0 ? 0 : a.Nmax;
    }
    if constexpr (!SK) {
        const int n_total = SPARSE ? a.top_k : n_b;
        nsplit_b = n_total > 0 ? (n_total + a.chunk - 1) / a.chunk : 1;
        if (split >= nsplit_b)
            return;
        t0 = split * a.chunk;
        t1 = min(t0 + a.chunk, n_total);
    }
    // rounds of this CTA: t0, t0 + step, ... below t1 (interleaved: every
    // nsplit_b-th round of the pair, starting at round `split`)
    int step = kTokPerRound;
    if constexpr (!SPARSE && !SK && !DB) {
        if (a.interleave) {
            t0 = split * kTokPerRound;
            t1 = n_b;
            step = nsplit_b * kTokPerRound;
        }
    }
    const size_t bg = (size_t)b * a.Hkv + g;
    const uint16_t *kbase = a.k + bg * (size_t)a.Nmax * kHeadDim;
    const uint16_t *vbase = a.v + bg * (size_t)a.Nmax * kHeadDim;

    if constexpr (SELECT) {
        for (int i = tid; i < kSelectBins; i += NT)
            sm_hist[i] = 0u;
        __syncthreads();
    }
    if constexpr (SPARSE) {
        if (a.idx_dep)
            pdl_wait();
        const int32_t *ip = a.idx + bg * (size_t)a.top_k;
        for (int j = tid; j < t1 - t0; j += NT) {
            int rr = ip[t0 + j];
            if (rr < -1 || rr >= n_b) {
                atomicOr(a.status, kFlagIndexOutOfRange);
                rr = -1;
            }
            sm_rows[j] = rr;
        }
        __syncthreads();
    }
    auto row_of = [&](int t) { return t < t1 ? (SPARSE ? sm_rows[t - t0] : t) : -1; };

    // This warp's 16 tokens of the round at `base`: K of tokens r, r + 8
    // (dims 16j + 4c .. +3 for k-step j); V of tokens 2c, 2c+1, 2c+8, 2c+9
    // (dims 8r..8r+7 and 64+8r..64+8r+7).
    auto load = [&](int base, uint2 (&kq)[2][8], uint4 (&vv)[4][2]) {
        const int tw = base + warp * 16;
        const int rk[2] = {row_of(tw + r), row_of(tw + r + 8)};
        const int rv[4] = {row_of(tw + 2 * c), row_of(tw + 2 * c + 1), row_of(tw + 2 * c + 8),
                           row_of(tw + 2 * c + 9)};
#pragma unroll
        for (int t = 0; t < 2; ++t)
#pragma unroll
            for (int j = 0; j < 8; ++j)
                kq[t][j] = rk[t] >= 0 ? ldg8(kbase + (size_t)rk[t] * kHeadDim + 16 * j + 4 * c)
                                      : make_uint2(0u, 0u);
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int t = 0; t < 4; ++t)
                vv[t][i] = rv[t] >= 0 ? ldg16(vbase + (size_t)rv[t] * kHeadDim + 64 * i + 8 * r)
                                      : make_uint4(0u, 0u, 0u, 0u);
    };
    // L2 prefetch of this warp's round (two calls of 8 tokens)
    auto prefetch = [&](int base) {
        prefetch_round_l2(kbase, vbase, base + warp * 16, lane, row_of);
        prefetch_round_l2(kbase, vbase, base + warp * 16 + 8, lane, row_of);
    };
    uint2 kq0[2][8], kq1[2][8];
    uint4 vv0[4][2], vv1[4][2];
    load(t0, kq0, vv0);  // the cache is never written by a kernel of the step
    if constexpr (DB)
        load(t0 + kTokPerRound, kq1, vv1);
    // full layers: rounds 1 .. prefetch go to L2 now, later rounds `prefetch`
    // ahead of use
    const int pf = SPARSE ? 0 : a.prefetch;
    for (int d = 1; d <= pf; ++d)
        prefetch(t0 + d * step);
    pdl_wait();

    // q of head r (heads >= G are zero columns): dims 16j + 4c .. +3.
    uint2 qf[8];
#pragma unroll
    for (int j = 0; j < 8; ++j)
        qf[j] = r < G ? *reinterpret_cast<const uint2 *>(
                            a.q + ((size_t)b * a.Hq + (size_t)g * G + r) * kHeadDim + 16 * j + 4 * c)
                      : make_uint2(0u, 0u);

    const float c2 = a.scale * kLog2e;
    float m[2] = {-CUDART_INF_F, -CUDART_INF_F};  // heads 2c, 2c+1 (replicated over r)
    float l[2] = {0.0f, 0.0f};
    // m-tile i holds dims vdim(i) (0, 1: heads 2c, 2c+1) and vdim(i) + 1 (2, 3),
    // vdim(i) = (i < 4 ? 8r : 64 + 8r) + 2 (i % 4)
    float o[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j)
            o[i][j] = 0.0f;

    auto round = [&](int base, const uint2 (&kq)[2][8], const uint4 (&vv)[4][2]) {
        const int tw = base + warp * 16;
        // s[0], s[1]: token r, heads 2c, 2c+1; s[2], s[3]: token r + 8
        float s[4] = {0.0f, 0.0f, 0.0f, 0.0f}, s_odd[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
        for (int j = 0; j < 8; j += 2) {  // two chains of 4 dependent MMAs
            mma_bf16(s, kq[0][j].x, kq[1][j].x, kq[0][j].y, kq[1][j].y, qf[j].x, qf[j].y);
            mma_bf16(s_odd, kq[0][j + 1].x, kq[1][j + 1].x, kq[0][j + 1].y, kq[1][j + 1].y,
                     qf[j + 1].x, qf[j + 1].y);
        }
#pragma unroll
        for (int e = 0; e < 4; ++e)
            s[e] += s_odd[e];
        const bool ok[2] = {row_of(tw + r) >= 0, row_of(tw + r + 8) >= 0};

        if constexpr (SELECT) {
            // selection scores of tokens tw + r, tw + r + 8: the group's summed
            // scaled logits (lane c = 0 stores the first, c = 1 the second)
#pragma unroll
            for (int t = 0; t < 2; ++t) {
                float sc = (2 * c < G ? s[2 * t] * a.scale : 0.0f) +
                           (2 * c + 1 < G ? s[2 * t + 1] * a.scale : 0.0f);
                sc += __shfl_xor_sync(kFull, sc, 1);
                sc += __shfl_xor_sync(kFull, sc, 2);
                const int tok = tw + r + 8 * t;
                if (c == t && tok < t1) {
                    a.scores[bg * (size_t)a.Nmax + tok] = sc;
                    atomicAdd(&sm_hist[order_key(sc) >> (32 - kSelectBits)], 1u);
                }
            }
        }

        // online softmax of heads 2c, 2c+1 over the warp's 16 tokens
        float p[2][2];  // [head 2c + e][token r, r + 8]
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const bool head = 2 * c + e < G;
            const float x0 = (ok[0] && head) ? s[e] * c2 : -CUDART_INF_F;
            const float x1 = (ok[1] && head) ? s[2 + e] * c2 : -CUDART_INF_F;
            float mx = fmaxf(x0, x1);
            mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 4));
            mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 8));
            mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 16));
            const float m_new = fmaxf(m[e], mx);
            float alpha = 1.0f;
            p[e][0] = p[e][1] = 0.0f;
            if (m_new != -CUDART_INF_F) {  // uniform over the 8 lanes of this head
                alpha = safe_exp2_diff(m[e], m_new);
                p[e][0] = (x0 == -CUDART_INF_F) ? 0.0f : exp2f(x0 - m_new);
                p[e][1] = (x1 == -CUDART_INF_F) ? 0.0f : exp2f(x1 - m_new);
            }
            float ps = p[e][0] + p[e][1];
            ps += __shfl_xor_sync(kFull, ps, 4);
            ps += __shfl_xor_sync(kFull, ps, 8);
            ps += __shfl_xor_sync(kFull, ps, 16);
            if (m_new != -CUDART_INF_F) {
                l[e] = l[e] * alpha + ps;
                m[e] = m_new;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    o[i][e] *= alpha;
                    o[i][e + 2] *= alpha;
                }
            }
        }

        // P^T fragment: P[token 2c + 8t][head r], P[token 2c + 1 + 8t][head r],
        // held by lanes (row 2c / 2c+1, quad r / 2) in p[r & 1][t]
        const int src0 = 8 * c + (r >> 1), src1 = 8 * c + 4 + (r >> 1);
        uint32_t pb[2][3];
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            const float a0p = __shfl_sync(kFull, p[0][t], src0), a1p = __shfl_sync(kFull, p[1][t], src0);
            const float b0p = __shfl_sync(kFull, p[0][t], src1), b1p = __shfl_sync(kFull, p[1][t], src1);
            float pt0 = (r & 1) ? a1p : a0p;
            float pt1 = (r & 1) ? b1p : b0p;
#pragma unroll
            for (int k = 0; k < 3; ++k) {  // p = p1 + p2 + p3 in bf16
                const __nv_bfloat16 h0 = __float2bfloat16_rn(pt0), h1 = __float2bfloat16_rn(pt1);
                pb[t][k] =
                    (uint32_t)__bfloat16_as_ushort(h0) | ((uint32_t)__bfloat16_as_ushort(h1) << 16);
                pt0 -= __bfloat162float(h0);
                pt1 -= __bfloat162float(h1);
            }
        }
        // O += V^T P^T, one m-tile of 16 dims at a time, k = tokens 2c, 2c+1,
        // 2c+8, 2c+9
        uint32_t lo[8], hi[8], lo8[8], hi8[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t w0 = word2(vv[0], i), w1 = word2(vv[1], i);
            const uint32_t w8 = word2(vv[2], i), w9 = word2(vv[3], i);
            lo[i] = prmt(w0, w1, 0x5410u);
            hi[i] = prmt(w0, w1, 0x7632u);
            lo8[i] = prmt(w8, w9, 0x5410u);
            hi8[i] = prmt(w8, w9, 0x7632u);
        }
#pragma unroll
        for (int k = 0; k < 3; ++k)  // consecutive MMAs go to different tiles
#pragma unroll
            for (int i = 0; i < 8; ++i)
                mma_bf16(o[i], lo[i], hi[i], lo8[i], hi8[i], pb[0][k], pb[1][k]);
    };

    if constexpr (DB) {
        // rounds in pairs: buffer 0 holds even rounds, buffer 1 odd ones; each
        // buffer is refilled (two rounds ahead) right after its round's arithmetic
        for (int base = t0; base < t1; base += 2 * kTokPerRound) {
            if (pf > 0)
                prefetch(base + pf * kTokPerRound);
            round(base, kq0, vv0);
            load(base + 2 * kTokPerRound, kq0, vv0);
            if (base + kTokPerRound < t1) {
                if (pf > 0)
                    prefetch(base + (pf + 1) * kTokPerRound);
                round(base + kTokPerRound, kq1, vv1);
                load(base + 3 * kTokPerRound, kq1, vv1);
            }
        }
    } else {
        // with early_trigger the next kernel may launch from the start of
        // round n_rounds - early_trigger of this CTA
        const int n_rounds = t1 > t0 ? (t1 - t0 + step - 1) / step : 0;
        const int trig = (!SK && a.early_trigger > 0) ? max(n_rounds - a.early_trigger, 0) : -1;
        if (trig == 0)
            pdl_launch_dependents();
        if (t0 < t1)
            round(t0, kq0, vv0);
        int ri = 1;
        for (int base = t0 + step; base < t1; base += step, ++ri) {
            if (ri == trig)
                pdl_launch_dependents();
            if (pf > 0)
                prefetch(base + pf * step);
            load(base, kq0, vv0);
            round(base, kq0, vv0);
        }
    }

    pdl_launch_dependents();

    // this warp's partial into shared memory (dims back in natural order)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        const int h = 2 * c + e;
        if (h < G) {
            if (r == 0) {
                sm_m[warp][h] = m[e];
                sm_l[warp][h] = l[e];
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int d = (i < 4 ? 8 * r : 64 + 8 * r) + 2 * (i & 3);
                sm_o[warp][h][d] = o[i][e];
                sm_o[warp][h][d + 1] = o[i][e + 2];
            }
        }
    }
    __syncthreads();
    if constexpr (SELECT) {
        unsigned *gh = a.hist + bg * kSelectBins;
        for (int i = tid; i < kSelectBins; i += NT)
            if (sm_hist[i])
                atomicAdd(&gh[i], sm_hist[i]);
    }
    if (tid < G) {
        const int h = tid;
        float M = -CUDART_INF_F;
        for (int w = 0; w < NW; ++w)
            M = fmaxf(M, sm_m[w][h]);
        float L = 0.0f;
        for (int w = 0; w < NW; ++w) {
            const float wt = safe_exp2_diff(sm_m[w][h], M);
            sm_w[w][h] = wt;
            L += sm_l[w][h] * wt;
        }
        sm_M[h] = M;
        sm_L[h] = L;
    }
    __syncthreads();
    const size_t out_row0 = (size_t)b * a.Hq + (size_t)g * G;
    finish_splits<G, NW, NT>(a, sm_o, sm_w, sm_M, sm_L, &sm_last, bg, split, nsplit_b, out_row0);
    }  // segments
}

template <typename Kern>
cudaError_t launch_kernel(Kern kern, int threads, const AttnArgs &a, int batch, bool pdl,
                          cudaStream_t stream)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)a.nsplit, (unsigned)a.Hkv, (unsigned)batch);
    cfg.blockDim = dim3(threads);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, a);
}

template <typename Kern>
int occupancy(Kern kern, int threads)
{
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, threads, 0) != cudaSuccess)
        return 1;
    return n > 0 ? n : 1;
}

// The ring kernel's shared-memory opt-in, once per device.
template <int G>
cudaError_t configure_ring()
{
    static bool configured[64] = {false};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev >= 0 && dev < 64 && configured[dev])
        return cudaSuccess;
    e = cudaFuncSetAttribute(attention_mma_ring_kernel<G>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kRingSmemBytes);
    if (e == cudaSuccess && dev >= 0 && dev < 64)
        configured[dev] = true;
    return e;
}

// tokens: 8 (attention_mma_kernel), 16 (attention_mma16_kernel, one round in
// flight per warp), 32 (attention_mma16_kernel, two rounds in flight) or, for
// sparse layers, 64 (attention_mma_ring_kernel, rounds staged in shared memory).
// a.sk_ctas > 0 (sparse, tokens 16 or 32): the stream-K partition over a 1D
// grid of a.sk_ctas CTAs for a.sk_units (batch row, KV head) pairs (partials
// with a stride of a.nsplit per pair).
template <int G, bool SPARSE, bool SELECT>
cudaError_t launch_mma_one(int tokens, const AttnArgs &a, int batch, bool pdl, cudaStream_t st)
{
    if constexpr (SPARSE) {
        if (a.sk_ctas > 0) {
            const AttnArgs &sk = a;
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3((unsigned)a.sk_ctas);
            cfg.blockDim = dim3(kMma16Threads);
            cfg.stream = st;
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
            attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            return tokens == 32
                       ? cudaLaunchKernelEx(&cfg, attention_mma16_kernel<G, true, false, true, true>, sk)
                       : cudaLaunchKernelEx(&cfg, attention_mma16_kernel<G, true, false, false, true>, sk);
        }
    }
    if constexpr (SPARSE) {
        if (tokens == 64) {
            const cudaError_t e = configure_ring<G>();
            if (e != cudaSuccess)
                return e;
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3((unsigned)a.nsplit, (unsigned)a.Hkv, (unsigned)batch);
            cfg.blockDim = dim3(kAttnThreads);
            cfg.dynamicSmemBytes = kRingSmemBytes;
            cfg.stream = st;
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
            attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            return cudaLaunchKernelEx(&cfg, attention_mma_ring_kernel<G>, a);
        }
    }
    if (tokens == 32)
        return launch_kernel(attention_mma16_kernel<G, SPARSE, SELECT, true>, kMma16Threads, a,
                             batch, pdl, st);
    if (tokens == 16)
        return launch_kernel(attention_mma16_kernel<G, SPARSE, SELECT, false>, kMma16Threads, a,
                             batch, pdl, st);
    return launch_kernel(attention_mma_kernel<G, SPARSE, SELECT>, kAttnThreads, a, batch, pdl, st);
}

template <int G, bool SPARSE, bool SELECT>
int mma_occupancy_one(int tokens)
{
    if (SPARSE && tokens == 64) {
        if (configure_ring<G>() != cudaSuccess)
            return 1;
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, attention_mma_ring_kernel<G>,
                                                          kAttnThreads, kRingSmemBytes) != cudaSuccess)
            return 1;
        return n > 0 ? n : 1;
    }
    if (tokens == 32)
        return occupancy(attention_mma16_kernel<G, SPARSE, SELECT, true>, kMma16Threads);
    if (tokens == 16)
        return occupancy(attention_mma16_kernel<G, SPARSE, SELECT, false>, kMma16Threads);
    return occupancy(attention_mma_kernel<G, SPARSE, SELECT>, kAttnThreads);
}

template <int G>
cudaError_t launch_mma_g(bool sparse, bool select, int tokens, const AttnArgs &a, int batch,
                         bool pdl, cudaStream_t st)
{
    if (sparse)
        return launch_mma_one<G, true, false>(tokens, a, batch, pdl, st);
    if (select)
        return launch_mma_one<G, false, true>(tokens, a, batch, pdl, st);
    return launch_mma_one<G, false, false>(tokens, a, batch, pdl, st);
}

template <int G>
int mma_occupancy_g(bool sparse, bool select, int tokens)
{
    return sparse ? mma_occupancy_one<G, true, false>(tokens)
                  : (select ? mma_occupancy_one<G, false, true>(tokens)
                            : mma_occupancy_one<G, false, false>(tokens));
}

}  // namespace

bool mma_supported(int G) { return G == 4 || G == 8; }

cudaError_t launch_attention_mma(int G, bool sparse, bool select, int tokens, const AttnArgs &a,
                                 int batch, bool pdl, cudaStream_t stream)
{
    if (G == 4)
        return launch_mma_g<4>(sparse, select, tokens, a, batch, pdl, stream);
    if (G == 8)
        return launch_mma_g<8>(sparse, select, tokens, a, batch, pdl, stream);
    return cudaErrorInvalidValue;
}

int attention_mma_ctas_per_sm(int G, bool sparse, bool select, int tokens)
{
    if (G == 4)
        return mma_occupancy_g<4>(sparse, select, tokens);
    if (G == 8)
        return mma_occupancy_g<8>(sparse, select, tokens);
    return 1;
}

}  // namespace td
