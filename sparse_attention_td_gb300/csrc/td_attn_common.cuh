// td_attn_common.cuh -- device helpers shared by the attention kernels
// (register/shared-memory paths in td_attn.cu, tensor-core path in
// td_attn_mma.cu): launch-dependency waits, the score key, L2 prefetch, and
// the last stage of a split-K launch (a CTA's normalised partial result, the
// split merge by the last-arriving CTA of a (batch row, KV head)).  The top-k
// kernels (td_topk.cu) use the same score key and waits.
#pragma once

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
// Pairs of consecutive dims as float2 (2j, 2j+1), for the packed fp32 pipe
// (one fma.rn.f32x2 does two IEEE fmas).
__device__ __forceinline__ void unpack8x2(const uint4 v, float2 (&f)[4])
{
    f[0] = make_float2(__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xffff0000u));
    f[1] = make_float2(__uint_as_float(v.y << 16), __uint_as_float(v.y & 0xffff0000u));
    f[2] = make_float2(__uint_as_float(v.z << 16), __uint_as_float(v.z & 0xffff0000u));
    f[3] = make_float2(__uint_as_float(v.w << 16), __uint_as_float(v.w & 0xffff0000u));
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
// L2 prefetch of the K and V rows a warp takes in one round: its 8 tokens
// starting at `tw`, one 128-byte line per lane (lanes 0-15 K, 16-31 V, two
// lines per row).  `row_of(t)` gives a token's cache row, or -1 to skip it.
template <typename RowOf>
__device__ __forceinline__ void prefetch_round_l2(const uint16_t *kbase, const uint16_t *vbase,
                                                  int tw, int lane, RowOf row_of)
{
    const int row = row_of(tw + ((lane >> 1) & 7));
    if (row >= 0) {
        const uint16_t *p = (lane < 16 ? kbase : vbase) + (size_t)row * kHeadDim + (lane & 1) * 64;
        asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
    }
}

// Stages a sparse CTA's index entries ip[t0 + j], j < count <= kMaxSparseChunk,
// into sm_rows[j]: -1 stays padding, anything else outside [0, n_b) is
// reported and skipped.  Every entry is requested before any is checked (the
// checks can report, so loads issued after them would wait for the previous
// checks), so the loads overlap one another and the caller's load of n_b.
// All NT threads call it; sm_rows is complete after the caller's barrier.
template <int NT>
__device__ __forceinline__ void stage_index_rows(const int32_t *ip, int t0, int count, int n_b,
                                                 uint32_t *status, int *sm_rows, int tid)
{
    constexpr int kPer = (kMaxSparseChunk + NT - 1) / NT;
    int rv[kPer];
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
        const int j = tid + u * NT;
        rv[u] = j < count ? __ldcg(ip + t0 + j) : -1;
    }
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
        const int j = tid + u * NT;
        if (j < count) {
            int rr = rv[u];
            if (rr < -1 || rr >= n_b) {
                atomicOr(status, kFlagIndexOutOfRange);
                rr = -1;
            }
            sm_rows[j] = rr;
        }
    }
}

__device__ __forceinline__ void pdl_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void pdl_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Order-preserving 32-bit key of a score, shared with the top-k kernel:
// larger float -> larger unsigned; -0.0 is mapped to +0.0 first so the two tie.
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


// Last stage of an attention CTA whose warps' partial results are merged in
// shared memory: sm_o[w][h][d] un-normalised outputs of warp w with weights
// sm_w[w][h] towards the CTA's running maximum sm_M[h] (log2 units) and
// denominator sm_L[h].  One split: write the normalised output.  Several:
// publish this split's partial and let the last CTA to arrive merge them all.
// All NT threads (NW warps) of the CTA call it.
template <int G, int NW = kAttnWarps, int NT = kAttnThreads>
__device__ __forceinline__ void finish_splits(const AttnArgs &a, const float (*sm_o)[G][kHeadDim],
                                              const float (*sm_w)[G], const float *sm_M,
                                              const float *sm_L, int *sm_last, size_t bg,
                                              int split, int nsplit_b, size_t out_row0)
{
    const int tid = threadIdx.x;
    if (nsplit_b == 1) {
        for (int e = tid; e < G * kHeadDim; e += NT) {
            const int h = e / kHeadDim, d = e % kHeadDim;
            float acc = 0.0f;
#pragma unroll
            for (int w = 0; w < NW; ++w)
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
    for (int e = tid; e < G * kHeadDim; e += NT) {
        const int h = e / kHeadDim, d = e % kHeadDim;
        float acc = 0.0f;
#pragma unroll
        for (int w = 0; w < NW; ++w)
            acc += sm_o[w][h][d] * sm_w[w][h];
        a.part_o[(pbase + h) * kHeadDim + d] = acc;
    }
    if (tid < G) {
        a.part_m[pbase + tid] = sm_M[tid];
        a.part_l[pbase + tid] = sm_L[tid];
    }
    // One thread takes the ticket with a release-acquire atomic at GPU scope:
    // the barrier orders the CTA's partial stores before it, and in the last
    // CTA the acquire plus the next barrier order the merge's loads after
    // every other split's release.  No thread-wide fences.
    __syncthreads();
    if (tid == 0) {
        unsigned ticket;
        asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], 1;"
                     : "=r"(ticket)
                     : "l"(a.tickets + bg)
                     : "memory");
        *sm_last = (ticket == (unsigned)(nsplit_b - 1));
    }
    __syncthreads();
    if (!*sm_last)
        return;

    // Last CTA of this (batch, KV head): merge all splits.  Each output
    // element's thread reads every split's (m, l) of its head and its own o
    // values as one batch of independent loads (chunks of kMergeChunk splits),
    // then reduces locally: one round trip instead of three with barriers.
    const size_t pb0 = bg * (size_t)a.nsplit * G;
    constexpr int kMergeChunk = 16;
    for (int e = tid; e < G * kHeadDim; e += NT) {
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

}  // namespace
}  // namespace td
