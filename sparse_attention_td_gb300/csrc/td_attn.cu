// td_attn.cu -- decode-step attention kernels for sm_103a.
//
// One kernel body serves both layer kinds of a TidalDecode decode step
// (TidalDecode paper review, §三 Figure 2):
//   * full attention (optionally with fused emission of the selection score),
//     streaming every cached token of a (batch, KV head) pair;
//   * PPSA sparse attention, gathering only the persisted token rows
//     (review §三 "Position Persistent Sparse Attention").
// Both compute A = q K^T / sqrt(d), H = softmax(A) V (review §三, PPSA
// formula) with an online softmax, split over the token axis
// (flash-decoding): each CTA owns one (split, KV head, batch row) and all G
// query heads of the KV head's group, so every K/V byte is read once.  The
// splits of a (batch, KV head) pair are merged by whichever CTA arrives last
// (an atomic ticket; nobody waits on anybody).
//
// The work is HBM-bound (about G flops per K/V byte), so there is no tensor
// core path: each half-warp reads one 256-byte K row and one V row with
// 16-byte loads (lane c holds dims 8c..8c+7), every thread keeps 4 tokens of
// K and V in flight, and dot products are reduced with warp shuffles.
#include <cooperative_groups.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math_constants.h>
#include <stdint.h>

#include "td_internal.h"

namespace td {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr float kLog2e = 1.4426950408889634f;

// bf16 -> fp32 is exact: a bf16 value is the upper half of its fp32 word.
__device__ __forceinline__ void unpack8(const uint4 v, float (&f)[8])
{
    f[0] = __uint_as_float(v.x << 16);
    f[1] = __uint_as_float(v.x & 0xffff0000u);
    f[2] = __uint_as_float(v.y << 16);
    f[3] = __uint_as_float(v.y & 0xffff0000u);
    f[4] = __uint_as_float(v.z << 16);
    f[5] = __uint_as_float(v.z & 0xffff0000u);
    f[6] = __uint_as_float(v.w << 16);
    f[7] = __uint_as_float(v.w & 0xffff0000u);
}

// K/V rows are read exactly once per layer: read-only path, no L1 allocation.
__device__ __forceinline__ uint4 load_row16(const uint16_t *p)
{
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// Programmatic dependent launch: the next kernel of the step may start while
// this one finishes.  Before pdl_wait() a kernel touches only what no kernel
// of the step writes (seq_lens, the K/V cache, and an index set produced
// earlier than by the kernel right before); after it, everything the
// previous kernel wrote (q in a full model, index set, scores, workspace) is
// complete and visible.
__device__ __forceinline__ void pdl_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void pdl_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Order-preserving 32-bit key of a score (as in the top-k kernel): larger
// float -> larger unsigned, -0.0 equal to +0.0.
__device__ __forceinline__ uint32_t order_key(float f)
{
    uint32_t u = __float_as_uint(f);
    if (u == 0x80000000u)
        u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float safe_exp2_diff(float x, float m)
{
    // exp2(x - m) with m = -inf meaning "no token seen yet" (weight 0)
    return (m == -CUDART_INF_F) ? 0.0f : exp2f(x - m);
}

__device__ __forceinline__ uint16_t f32_to_bf16_rn(float f)
{
    return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

namespace cg = cooperative_groups;

// CLUSTER: the splits of one (batch row, KV head) form a thread-block
// cluster (grid x = cluster x = splits) and are merged through distributed
// shared memory; otherwise through global partials and an arrival ticket.
template <int G, bool SPARSE, bool SELECT, bool CLUSTER>
__global__ void __launch_bounds__(kAttnThreads)
attention_kernel(const AttnArgs a)
{
    constexpr int U = kTokPerHalf;
    __shared__ float sm_m[kAttnWarps][G];
    __shared__ float sm_l[kAttnWarps][G];
    __shared__ float sm_w[kAttnWarps][G];
    __shared__ __align__(16) float sm_o[kAttnWarps][G][kHeadDim];
    __shared__ float sm_M[G];
    __shared__ float sm_L[G];
    __shared__ float sm_red[kAttnWarps][G];
    __shared__ int sm_rows[SPARSE ? kMaxSparseChunk : 1];
    __shared__ int sm_last;
    // selection layers: histogram of the scores' top 11 bits (the top-k kernel's first digit)
    __shared__ unsigned sm_hist[SELECT ? kSelectBins : 1];
    // per-split merge weights of the final combine; sm_o is dead by then
    static_assert(kMaxSplits <= kAttnWarps * kHeadDim, "sm_sw must fit in sm_o");
    float *sm_sw = &sm_o[0][0][0];

    const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int half = lane >> 4, c = lane & 15;

    int n_b = a.seq_lens[b];
    if (n_b < 0 || n_b > a.Nmax) {
        if (tid == 0)
            atomicOr(a.status, kFlagSeqLenOutOfRange);
        n_b = n_b < 0 ? 0 : a.Nmax;
    }
    const int n_total = SPARSE ? a.top_k : n_b;
    const int nsplit_b = n_total > 0 ? (n_total + a.chunk - 1) / a.chunk : 1;
    // A split past this row's work returns at once -- except in a cluster,
    // where it takes part in the merge with an empty range.
    const bool idle = split >= nsplit_b;
    if (idle && !CLUSTER)
        return;
    const int t0 = idle ? 0 : split * a.chunk;
    const int t1 = idle ? 0 : min(t0 + a.chunk, n_total);
    const size_t bg = (size_t)b * a.Hkv + g;
    const uint16_t *kbase = a.k + bg * (size_t)a.Nmax * kHeadDim + c * 8;
    const uint16_t *vbase = a.v + bg * (size_t)a.Nmax * kHeadDim + c * 8;

    if constexpr (SELECT) {
        for (int i = tid; i < kSelectBins; i += kAttnThreads)
            sm_hist[i] = 0u;
        __syncthreads();
    }
    if constexpr (SPARSE) {
        // The index set was computed earlier in the step, unless the kernel
        // right before this one produced it: then wait for that kernel first.
        if (a.idx_dep)
            pdl_wait();
        // Stage this split's persisted positions; -1 is padding, anything
        // else outside [0, n_b) is reported and skipped.
        const int32_t *ip = a.idx + bg * (size_t)a.top_k;
        for (int j = tid; j < t1 - t0; j += kAttnThreads) {
            int r = ip[t0 + j];
            if (r < -1 || r >= n_b) {
                atomicOr(a.status, kFlagIndexOutOfRange);
                r = -1;
            }
            sm_rows[j] = r;
        }
        __syncthreads();
    }

    // This half-warp's U tokens of the round starting at `base`: K and V rows
    // requested into registers (zero for tokens past the split or padding).
    auto load_round = [&](int base, uint4 (&kr)[U], uint4 (&vr)[U], bool (&ok)[U]) {
        const int tb = base + (warp * 2 + half) * U;
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int t = tb + u;
            int row = -1;
            if (t < t1)
                row = SPARSE ? sm_rows[t - t0] : t;
            ok[u] = row >= 0;
            kr[u] = ok[u] ? load_row16(kbase + (size_t)row * kHeadDim) : make_uint4(0u, 0u, 0u, 0u);
            vr[u] = ok[u] ? load_row16(vbase + (size_t)row * kHeadDim) : make_uint4(0u, 0u, 0u, 0u);
        }
    };
    // The cache is never written by a kernel of the step, so the first round
    // is requested before waiting for the previous kernel; q may come from it.
    uint4 kr0[U], vr0[U];
    bool ok0[U];
    load_round(t0, kr0, vr0, ok0);
    pdl_wait();

    // This lane's 8 dims of the group's G queries.
    float qf[G][8];
#pragma unroll
    for (int h = 0; h < G; ++h) {
        const uint4 qv = *reinterpret_cast<const uint4 *>(
            a.q + ((size_t)b * a.Hq + (size_t)g * G + h) * kHeadDim + c * 8);
        unpack8(qv, qf[h]);
    }

    const float c2 = a.scale * kLog2e;  // logits in log2 units for exp2
    float m[G], l[G], o[G][8];
#pragma unroll
    for (int h = 0; h < G; ++h) {
        m[h] = -CUDART_INF_F;
        l[h] = 0.0f;
#pragma unroll
        for (int i = 0; i < 8; ++i)
            o[h][i] = 0.0f;
    }

    // One round: scores, online softmax and P V for this half-warp's U tokens.
    auto round = [&](int base, const uint4 (&kr)[U], const uint4 (&vr)[U], const bool (&ok)[U]) {
        const int tb = base + (warp * 2 + half) * U;  // this half-warp's first token

        // q . k over this lane's 8 dims, then over the half-warp's 16 lanes.
        float dot[G][U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            float kf[8];
            unpack8(kr[u], kf);
#pragma unroll
            for (int h = 0; h < G; ++h) {
                float acc = 0.0f;
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    acc = fmaf(qf[h][i], kf[i], acc);
                dot[h][u] = acc;
            }
        }
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
            for (int u = 0; u < U; ++u)
#pragma unroll
                for (int off = 8; off >= 1; off >>= 1)
                    dot[h][u] += __shfl_xor_sync(kFull, dot[h][u], off);

        if constexpr (SELECT) {
            // Selection score of a KV head: the sum of its query heads'
            // scaled logits.  Lane c < U of the half stores token tb + c.
            float sc = 0.0f;
#pragma unroll
            for (int u = 0; u < U; ++u) {
                float s = 0.0f;
#pragma unroll
                for (int h = 0; h < G; ++h)
                    s += dot[h][u] * a.scale;
                if (c == u)
                    sc = s;
            }
            if (c < U && tb + c < t1) {
                a.scores[bg * (size_t)a.Nmax + tb + c] = sc;
                atomicAdd(&sm_hist[order_key(sc) >> (32 - kSelectBits)], 1u);
            }
        }

        // Online softmax over this round's U tokens, then P V.
        float p[G][U];
#pragma unroll
        for (int h = 0; h < G; ++h) {
            float t2[U];
            float mx = -CUDART_INF_F;
#pragma unroll
            for (int u = 0; u < U; ++u) {
                t2[u] = ok[u] ? dot[h][u] * c2 : -CUDART_INF_F;
                mx = fmaxf(mx, t2[u]);
            }
            const float m_new = fmaxf(m[h], mx);
            if (m_new != -CUDART_INF_F) {
                const float alpha = exp2f(m[h] - m_new);
                float ps = 0.0f;
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    p[h][u] = exp2f(t2[u] - m_new);
                    ps += p[h][u];
                }
                l[h] = l[h] * alpha + ps;
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    o[h][i] *= alpha;
                m[h] = m_new;
            } else {
#pragma unroll
                for (int u = 0; u < U; ++u)
                    p[h][u] = 0.0f;
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            float vf[8];
            unpack8(vr[u], vf);
#pragma unroll
            for (int h = 0; h < G; ++h)
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    o[h][i] = fmaf(p[h][u], vf[i], o[h][i]);
        }
    };
    if (t0 < t1)
        round(t0, kr0, vr0, ok0);
    for (int base = t0 + kTokPerRound; base < t1; base += kTokPerRound) {
        uint4 kr[U], vr[U];
        bool ok[U];
        load_round(base, kr, vr, ok);
        round(base, kr, vr, ok);
    }

    pdl_launch_dependents();  // the next kernel's CTAs may start requesting their cache rows

    // Merge the two half-warps, then the 8 warps, of this CTA.
#pragma unroll
    for (int h = 0; h < G; ++h) {
        const float m_o = __shfl_xor_sync(kFull, m[h], 16);
        const float l_o = __shfl_xor_sync(kFull, l[h], 16);
        const float m_new = fmaxf(m[h], m_o);
        const float sa = safe_exp2_diff(m[h], m_new);
        const float so = safe_exp2_diff(m_o, m_new);
        l[h] = l[h] * sa + l_o * so;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float oo = __shfl_xor_sync(kFull, o[h][i], 16);
            o[h][i] = o[h][i] * sa + oo * so;
        }
        m[h] = m_new;
    }
    if (half == 0) {
#pragma unroll
        for (int h = 0; h < G; ++h) {
            if (c == 0) {
                sm_m[warp][h] = m[h];
                sm_l[warp][h] = l[h];
            }
            float4 *dst = reinterpret_cast<float4 *>(&sm_o[warp][h][c * 8]);
            dst[0] = make_float4(o[h][0], o[h][1], o[h][2], o[h][3]);
            dst[1] = make_float4(o[h][4], o[h][5], o[h][6], o[h][7]);
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

    const size_t out_row0 = (size_t)b * a.Hq + (size_t)g * G;  // first query head of the group
    if constexpr (CLUSTER) {
        // This split's partial (un-normalised o, M, L) stays in shared
        // memory: o in sm_o[0], M and L in sm_M / sm_L.
        constexpr int PER = (G * kHeadDim + kAttnThreads - 1) / kAttnThreads;
        float part[PER];
#pragma unroll
        for (int j = 0; j < PER; ++j) {
            const int e = tid + j * kAttnThreads;
            part[j] = 0.0f;
            if (e < G * kHeadDim) {
                const int h = e / kHeadDim, d = e % kHeadDim;
#pragma unroll
                for (int w = 0; w < kAttnWarps; ++w)
                    part[j] += sm_o[w][h][d] * sm_w[w][h];
            }
        }
        __syncthreads();
#pragma unroll
        for (int j = 0; j < PER; ++j) {
            const int e = tid + j * kAttnThreads;
            if (e < G * kHeadDim)
                sm_o[0][e / kHeadDim][e % kHeadDim] = part[j];
        }
        cg::cluster_group cluster = cg::this_cluster();
        cluster.sync();  // every split's partial is in its shared memory
        if (split == 0) {
            const int ns = (int)cluster.num_blocks();
            __shared__ float sm_cw[kMaxClusterSplits][G];  // merge weight of split r, head h
            if (tid < G) {
                float M = -CUDART_INF_F;
                for (int r = 0; r < ns; ++r)
                    M = fmaxf(M, *cluster.map_shared_rank(&sm_M[tid], r));
                float L = 0.0f;
                for (int r = 0; r < ns; ++r) {
                    const float wt = safe_exp2_diff(*cluster.map_shared_rank(&sm_M[tid], r), M);
                    sm_cw[r][tid] = wt;
                    L += *cluster.map_shared_rank(&sm_L[tid], r) * wt;
                }
                sm_red[0][tid] = L;
            }
            __syncthreads();
            for (int e = tid; e < G * kHeadDim; e += kAttnThreads) {
                const int h = e / kHeadDim, d = e % kHeadDim;
                float acc = 0.0f;
                for (int r = 0; r < ns; ++r)
                    acc += sm_cw[r][h] * *cluster.map_shared_rank(&sm_o[0][h][d], r);
                const float L = sm_red[0][h];
                const float val = L > 0.0f ? acc / L : 0.0f;
                a.out[(out_row0 + h) * kHeadDim + d] = f32_to_bf16_rn(val);
                if (a.out_f32)
                    a.out_f32[(out_row0 + h) * kHeadDim + d] = val;
            }
        }
        cluster.sync();  // keep every split's shared memory alive until split 0 has read it
        return;
    }
    if (nsplit_b == 1) {
        for (int e = tid; e < G * kHeadDim; e += kAttnThreads) {
            const int h = e / kHeadDim, d = e % kHeadDim;
            float acc = 0.0f;
#pragma unroll
            for (int w = 0; w < kAttnWarps; ++w)
                acc += sm_o[w][h][d] * sm_w[w][h];
            const float L = sm_L[h];
            const float val = L > 0.0f ? acc / L : 0.0f;
            a.out[(out_row0 + h) * kHeadDim + d] = f32_to_bf16_rn(val);
            if (a.out_f32)
                a.out_f32[(out_row0 + h) * kHeadDim + d] = val;
        }
        return;
    }

    // Several splits: publish this split's partial result.
    const size_t pbase = (bg * (size_t)a.nsplit + split) * G;
    for (int e = tid; e < G * kHeadDim; e += kAttnThreads) {
        const int h = e / kHeadDim, d = e % kHeadDim;
        float acc = 0.0f;
#pragma unroll
        for (int w = 0; w < kAttnWarps; ++w)
            acc += sm_o[w][h][d] * sm_w[w][h];
        a.part_o[(pbase + h) * kHeadDim + d] = acc;
    }
    if (tid < G) {
        a.part_m[pbase + tid] = sm_M[tid];
        a.part_l[pbase + tid] = sm_L[tid];
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        const unsigned ticket = atomicAdd(&a.tickets[bg], 1u);
        sm_last = (ticket == (unsigned)(nsplit_b - 1));
    }
    __syncthreads();
    if (!sm_last)
        return;
    __threadfence();

    // Last CTA of this (batch, KV head): merge all splits.  Each output
    // element's thread reads every split's (m, l) of its head and its own o
    // values as one batch of independent loads (chunks of kMergeChunk splits),
    // then reduces locally: one round trip instead of three with barriers.
    const size_t pb0 = bg * (size_t)a.nsplit * G;
    constexpr int kMergeChunk = 16;
    for (int e = tid; e < G * kHeadDim; e += kAttnThreads) {
        const int h = e / kHeadDim, d = e % kHeadDim;
        float M = -CUDART_INF_F, L = 0.0f, acc = 0.0f;
        for (int s0 = 0; s0 < nsplit_b; s0 += kMergeChunk) {
            float mv[kMergeChunk], lv[kMergeChunk], ov[kMergeChunk];
#pragma unroll
            for (int j = 0; j < kMergeChunk; ++j) {
                const int s = s0 + j;
                mv[j] = -CUDART_INF_F;
                lv[j] = 0.0f;
                ov[j] = 0.0f;
                if (s < nsplit_b) {
                    const size_t ps = pb0 + (size_t)s * G + h;
                    mv[j] = __ldcg(&a.part_m[ps]);
                    lv[j] = __ldcg(&a.part_l[ps]);
                    ov[j] = __ldcg(&a.part_o[ps * kHeadDim + d]);
                }
            }
            float Mc = M;
#pragma unroll
            for (int j = 0; j < kMergeChunk; ++j)
                Mc = fmaxf(Mc, mv[j]);
            const float r = safe_exp2_diff(M, Mc);  // rescale what earlier chunks added
            acc *= r;
            L *= r;
#pragma unroll
            for (int j = 0; j < kMergeChunk; ++j) {
                const float wt = safe_exp2_diff(mv[j], Mc);
                acc += wt * ov[j];
                L += wt * lv[j];
            }
            M = Mc;
        }
        const float val = L > 0.0f ? acc / L : 0.0f;
        a.out[(out_row0 + h) * kHeadDim + d] = f32_to_bf16_rn(val);
        if (a.out_f32)
            a.out_f32[(out_row0 + h) * kHeadDim + d] = val;
    }
    if (tid == 0)
        a.tickets[bg] = 0u;  // ready for the next launch on this workspace
}

int g_carveout = -1;  // preferred shared-memory carveout (percent) for the attention kernels

template <int G, bool SPARSE, bool SELECT, bool CLUSTER>
cudaError_t launch_one(const AttnArgs &a, int batch, cudaStream_t stream)
{
    if (g_carveout >= 0)
        cudaFuncSetAttribute(attention_kernel<G, SPARSE, SELECT, CLUSTER>,
                             cudaFuncAttributePreferredSharedMemoryCarveout, g_carveout);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)a.nsplit, (unsigned)a.Hkv, (unsigned)batch);
    cfg.blockDim = dim3(kAttnThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    int nattr = 1;
    if (CLUSTER) {
        if (a.nsplit > 8) {  // beyond the portable cluster size
            cudaError_t e = cudaFuncSetAttribute(attention_kernel<G, SPARSE, SELECT, CLUSTER>,
                                                 cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
            if (e != cudaSuccess)
                return e;
        }
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = (unsigned)a.nsplit;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        nattr = 2;
    }
    cfg.attrs = attr;
    cfg.numAttrs = nattr;
    return cudaLaunchKernelEx(&cfg, attention_kernel<G, SPARSE, SELECT, CLUSTER>, a);
}

template <int G, bool SPARSE, bool SELECT>
int occupancy_one()
{
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, attention_kernel<G, SPARSE, SELECT, false>,
                                                      kAttnThreads, 0) != cudaSuccess)
        return 1;
    return n > 0 ? n : 1;
}

}  // namespace

void set_attention_carveout(int percent) { g_carveout = percent; }

cudaError_t launch_attention(int G, bool sparse, bool select, bool cluster, const AttnArgs &a,
                             int batch, cudaStream_t stream)
{
#define TD_DISPATCH_G(GG)                                                             \
    case GG:                                                                          \
        if (sparse)                                                                   \
            return cluster ? launch_one<GG, true, false, true>(a, batch, stream)      \
                           : launch_one<GG, true, false, false>(a, batch, stream);    \
        if (select)                                                                   \
            return cluster ? launch_one<GG, false, true, true>(a, batch, stream)      \
                           : launch_one<GG, false, true, false>(a, batch, stream);    \
        return cluster ? launch_one<GG, false, false, true>(a, batch, stream)         \
                       : launch_one<GG, false, false, false>(a, batch, stream);
    switch (G) {
        TD_DISPATCH_G(1)
        TD_DISPATCH_G(2)
        TD_DISPATCH_G(4)
        TD_DISPATCH_G(8)
    default:
        return cudaErrorInvalidValue;
    }
#undef TD_DISPATCH_G
}

int attention_ctas_per_sm(int G, bool sparse, bool select)
{
#define TD_OCC_G(GG)                                                      \
    case GG:                                                              \
        if (sparse)                                                       \
            return occupancy_one<GG, true, false>();                      \
        if (select)                                                       \
            return occupancy_one<GG, false, true>();                      \
        return occupancy_one<GG, false, false>();
    switch (G) {
        TD_OCC_G(1)
        TD_OCC_G(2)
        TD_OCC_G(4)
        TD_OCC_G(8)
    default:
        return 1;
    }
#undef TD_OCC_G
}

}  // namespace td
