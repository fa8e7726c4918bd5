// td_attn_mma.cu -- grouped-query attention on the tensor cores (G = 4, 8).
//
// The same layer math as td_attn.cu (TidalDecode paper review, §三:
// A = q K^T / sqrt(d), H = softmax(A) V, split over the token axis, full or
// over the persisted positions), with both contractions over a KV head's G
// query heads done by mma.sync m16n8k16 (bf16 inputs, fp32 accumulation):
//   S[token][head] = K Q^T   (M = tokens, N = heads padded to 8, K = dims)
//   O[dim][head]  += V^T P^T (M = dims,   N = heads,              K = tokens)
// A warp takes 8 tokens per round (the upper 8 MMA rows stay zero), a CTA of
// 8 warps 64, as in the CUDA-core kernels, and the splits merge the same way.
//
// Fragments come straight from global memory.  The dot product does not care
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

__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
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
        float s[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
        for (int j = 0; j < 8; ++j)
            mma_bf16(s, kq[j].x, 0u, kq[j].y, 0u, qf[j].x, qf[j].y);
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
        // O += V^T P^T, one m-tile of 16 dims at a time
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t w0 = word2(v0, i), w1 = word2(v1, i);
            const uint32_t lo = prmt(w0, w1, 0x5410u);  // dim vdim(i) of tokens 2c, 2c+1
            const uint32_t hi = prmt(w0, w1, 0x7632u);  // dim vdim(i) + 1
#pragma unroll
            for (int k = 0; k < 3; ++k)
                mma_bf16(o[i], lo, hi, 0u, 0u, pb[k], 0u);
        }
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

template <int G, bool SPARSE, bool SELECT>
cudaError_t launch_mma_one(const AttnArgs &a, int batch, bool pdl, cudaStream_t stream)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)a.nsplit, (unsigned)a.Hkv, (unsigned)batch);
    cfg.blockDim = dim3(kAttnThreads);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, attention_mma_kernel<G, SPARSE, SELECT>, a);
}

template <int G, bool SPARSE, bool SELECT>
int mma_occupancy_one()
{
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(
            &n, attention_mma_kernel<G, SPARSE, SELECT>, kAttnThreads, 0) != cudaSuccess)
        return 1;
    return n > 0 ? n : 1;
}

template <int G>
cudaError_t launch_mma_g(bool sparse, bool select, const AttnArgs &a, int batch, bool pdl,
                         cudaStream_t st)
{
    if (sparse)
        return launch_mma_one<G, true, false>(a, batch, pdl, st);
    if (select)
        return launch_mma_one<G, false, true>(a, batch, pdl, st);
    return launch_mma_one<G, false, false>(a, batch, pdl, st);
}

}  // namespace

bool mma_supported(int G) { return G == 4 || G == 8; }

cudaError_t launch_attention_mma(int G, bool sparse, bool select, const AttnArgs &a, int batch,
                                 bool pdl, cudaStream_t stream)
{
    if (G == 4)
        return launch_mma_g<4>(sparse, select, a, batch, pdl, stream);
    if (G == 8)
        return launch_mma_g<8>(sparse, select, a, batch, pdl, stream);
    return cudaErrorInvalidValue;
}

int attention_mma_ctas_per_sm(int G, bool sparse, bool select)
{
    if (G == 4)
        return sparse ? mma_occupancy_one<4, true, false>()
                      : (select ? mma_occupancy_one<4, false, true>() : mma_occupancy_one<4, false, false>());
    if (G == 8)
        return sparse ? mma_occupancy_one<8, true, false>()
                      : (select ? mma_occupancy_one<8, false, true>() : mma_occupancy_one<8, false, false>());
    return 1;
}

}  // namespace td
