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
// core path: each half-warp works on one 256-byte K row and one V row at a
// time (lane c holds dims 8c..8c+7) and dot products are reduced with warp
// shuffles.  The rows reach the registers one of two ways:
//   * register-streamed: 16-byte loads straight from HBM, 4 tokens of K and V
//     in flight per thread (32 KB per CTA);
//   * staged: asynchronous copies fill a ring of shared-memory stages of 64
//     tokens, completing on an mbarrier; the CTA computes on stage i while
//     stages i+1.. are in flight (up to 128 KB per CTA).  Full layers: one
//     bulk copy (cp.async.bulk) per K or V block of contiguous rows.  Sparse
//     layers: either per-thread cp.async of the 16-byte pieces each thread
//     reads (STAGED = 1), or TMA row gathers (cp.async.bulk.tensor
//     tile::gather4: four cache rows per copy, through a tensor map over the
//     cache's rows; STAGED = 2).
#include <cooperative_groups.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math_constants.h>
#include <stdint.h>

#include "td_attn_common.cuh"
#include "td_internal.h"

namespace td {
namespace {

// ---- staged path: bulk copies into shared memory completing on mbarriers
constexpr int kStageRowBytes = kHeadDim * 2;                   // one bf16 row
constexpr int kStageBytes = 2 * kTokPerRound * kStageRowBytes;  // K block + V block = 32 KB
constexpr int kStageTxPerToken = 2 * kStageRowBytes;
constexpr uint64_t kWaitLimitNs = 1000000000ull;  // a bounded mbarrier wait gives up after 1 s

// Ring depth per group size: two CTAs per SM where registers allow it.
__host__ __device__ constexpr int staged_stages(int G)
{
    return G <= 2 ? 3 : (G == 4 ? 2 : 4);
}

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, unsigned count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, unsigned bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(
                     smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ uint64_t global_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

// Bounded wait for the phase with the given parity to complete: polls until
// it has, or until `limit_ns` nanoseconds of the global timer have passed
// (then false).
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, unsigned parity,
                                          uint64_t limit_ns = kWaitLimitNs)
{
    const uint32_t addr = smem_u32(bar);
    const uint64_t t0 = global_ns();
    for (;;) {
        uint32_t done;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(done)
            : "r"(addr), "r"(parity)
            : "memory");
        if (done)
            return true;
        if (global_ns() - t0 > limit_ns)
            return false;
    }
}

// Four rows of a 2D tensor map (rows of 128 bf16 values, box 128 x 1) into
// 1024 contiguous bytes of shared memory, counted on `bar` in bytes.  The
// column coordinate is 0; a row coordinate past the map's last row reads
// zeros (and still counts its 256 bytes).
__device__ __forceinline__ void tma_gather4(void *dst, const TmaDesc *map, int r0, int r1, int r2,
                                            int r3, uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(smem_u32(dst)),
        "l"(map), "r"(0), "r"(r0), "r"(r1), "r"(r2), "r"(r3), "r"(smem_u32(bar))
        : "memory");
}

// Global -> shared bulk copy (16-byte aligned addresses, size a multiple of
// 16) whose completion is counted on `bar` in bytes.
__device__ __forceinline__ void bulk_copy_g2s(void *dst, const void *src, unsigned bytes,
                                              uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// 16-byte global -> shared copy through L2 only (cp.async.cg); completion is
// tracked per thread in commit groups.
__device__ __forceinline__ void cp_async16(void *dst, const void *src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src)
                 : "memory");
}

__device__ __forceinline__ void cp_async_commit()
{
    asm volatile("cp.async.commit_group;" ::: "memory");
}

template <int N>
__device__ __forceinline__ void cp_async_wait()
{
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ uint4 lds128(const unsigned char *p)
{
    return *reinterpret_cast<const uint4 *>(p);
}

namespace cg = cooperative_groups;

// CLUSTER: the splits of one (batch row, KV head) form a thread-block
// cluster (grid x = cluster x = splits) and are merged through distributed
// shared memory; otherwise through global partials and an arrival ticket.
// STAGED: 0 register-streamed; 1 rows reach shared memory by bulk copies
// (full layers) or per-thread cp.async (sparse layers); 2 (sparse layers
// only) by TMA row gathers (see the file comment).
template <int G, bool SPARSE, bool SELECT, bool CLUSTER, int STAGED>
// Register budgets: 64 (MHA, 4 CTAs per SM; 85 and 3 CTAs with selection), 128 (G = 2, 4:
// 2 CTAs per SM), 255 (G = 8).
__global__ void __launch_bounds__(kAttnThreads, G == 1 ? (SELECT ? 3 : 4) : (G <= 4 ? 2 : 1))
attention_kernel(const __grid_constant__ AttnArgs a)
{
    static_assert(STAGED != 2 || SPARSE, "TMA row gathers serve sparse layers");
    constexpr int U = kTokPerHalf;
    constexpr int S = staged_stages(G);
    extern __shared__ __align__(128) unsigned char sm_stage[];  // STAGED: [S][K rows | V rows]
    __shared__ __align__(8) uint64_t sm_full[STAGED ? S : 1];
    // a barrier nothing ever arrives on: with a.wait_test set, each CTA's
    // first stage wait polls it, so that the wait runs out (failure-report tests)
    __shared__ __align__(8) uint64_t sm_never;
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

    // (the length check reports once the index entries are requested)
    const int n_raw = a.seq_lens[b];
    const int n_b = n_raw < 0 ? 0 : (n_raw > a.Nmax ? a.Nmax : n_raw);
    const int n_total = SPARSE ? a.top_k : n_b;
    const int nsplit_b = n_total > 0 ? (n_total + a.chunk - 1) / a.chunk : 1;
    // A split past this row's work returns at once -- except in a cluster,
    // where it takes part in the merge with an empty range.
    const bool idle = split >= nsplit_b;
    if (idle && !CLUSTER) {
        if (tid == 0 && n_raw != n_b)
            atomicOr(a.status, kFlagSeqLenOutOfRange);
        return;
    }
    int t0 = idle ? 0 : split * a.chunk;
    int t1 = idle ? 0 : min(t0 + a.chunk, n_total);
    // register-streamed full layers, interleaved: this CTA takes every
    // nsplit_b-th 64-token round of the pair, starting at round `split`
    int step = kTokPerRound;
    if constexpr (!SPARSE && !STAGED && !CLUSTER) {
        if (a.interleave && !idle) {
            t0 = split * kTokPerRound;
            t1 = n_total;
            step = nsplit_b * kTokPerRound;
        }
    }
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
        // Stage this split's persisted positions once (every round reads
        // them from shared memory); -1 is padding, anything else outside
        // [0, n_b) is reported and skipped.
        stage_index_rows<kAttnThreads>(a.idx + bg * (size_t)a.top_k, t0, t1 - t0, n_b, a.status,
                                       sm_rows, tid);
        __syncthreads();
    }
    if (tid == 0 && n_raw != n_b)
        atomicOr(a.status, kFlagSeqLenOutOfRange);

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
    // Staged: stage `it` of the ring receives the 64 tokens starting at
    // t0 + it * 64.  Full layers: bulk copies of the K and V blocks, issued
    // by warp 0 and completing on the stage's mbarrier.
    const int n_it = t1 > t0 ? (t1 - t0 + kTokPerRound - 1) / kTokPerRound : 0;
    const uint16_t *krows = a.k + bg * (size_t)a.Nmax * kHeadDim;
    const uint16_t *vrows = a.v + bg * (size_t)a.Nmax * kHeadDim;
    auto issue_stage = [&](int it) {  // warp 0
        unsigned char *kst = sm_stage + (it % S) * kStageBytes;
        unsigned char *vst = kst + kStageBytes / 2;
        uint64_t *bar = &sm_full[it % S];
        const int base = t0 + it * kTokPerRound;
        if constexpr (SPARSE) {
            // STAGED == 2: the stage's 64 rows of K and of V, four per gather,
            // one gather per lane of warp 0 (lanes 0-15 K, 16-31 V); padding
            // and tokens past the split read the zero rows past the map.
            // Lane 0 announces the stage's bytes before any gather is issued.
            if (lane == 0)
                mbar_arrive_expect_tx(bar, (unsigned)kTokPerRound * kStageTxPerToken);
            __syncwarp();
            const int oob = a.tma_rows;  // first row past the map
            const int row0 = (int)(bg * (size_t)a.Nmax);
            auto grow = [&](int t) {
                const int p = t < t1 ? sm_rows[t - t0] : -1;
                return p >= 0 ? row0 + p : oob;
            };
            const int j = lane & 15;
            const int t = base + 4 * j;
            tma_gather4((lane < 16 ? kst : vst) + j * 4 * kStageRowBytes,
                        lane < 16 ? &a.tma_k : &a.tma_v, grow(t), grow(t + 1), grow(t + 2),
                        grow(t + 3), bar);
        } else {
            // contiguous rows: one copy for the K block, one for the V block
            const int n = min(kTokPerRound, t1 - base);
            if (lane == 0) {
                mbar_arrive_expect_tx(bar, (unsigned)n * kStageTxPerToken);
                bulk_copy_g2s(kst, krows + (size_t)base * kHeadDim, (unsigned)n * kStageRowBytes,
                              bar);
                bulk_copy_g2s(vst, vrows + (size_t)base * kHeadDim, (unsigned)n * kStageRowBytes,
                              bar);
            }
        }
    };

    // Sparse layers: each thread copies the 16-byte pieces it will read itself
    // (lane c of a half-warp: bytes 16c.. of the K and V rows of its U
    // tokens) with cp.async, one commit group per stage (empty past the end),
    // so a thread only ever waits for its own copies: no barrier in the loop.
    auto issue_rows_cp = [&](int it) {
        if (it < n_it) {
            unsigned char *kst = sm_stage + (it % S) * kStageBytes;
            unsigned char *vst = kst + kStageBytes / 2;
            const int slot0 = (warp * 2 + half) * U;
            const int tb = t0 + it * kTokPerRound + slot0;
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int t = tb + u;
                const int row = t < t1 ? sm_rows[t - t0] : -1;
                if (row >= 0) {
                    cp_async16(kst + (slot0 + u) * kStageRowBytes + c * 16,
                                krows + (size_t)row * kHeadDim + c * 8);
                    cp_async16(vst + (slot0 + u) * kStageRowBytes + c * 16,
                                vrows + (size_t)row * kHeadDim + c * 8);
                }
            }
        }
        cp_async_commit();
    };

    // No attention or top-k kernel writes the cache (a step's KV append runs
    // before its first attention kernel, which is not overlapped with it), so
    // the first round (register-streamed) or the first S stages (staged) are
    // requested before waiting for the previous kernel; q may come from it.
    uint4 kr0[U], vr0[U];
    bool ok0[U];
    if constexpr (STAGED == 1 && SPARSE) {
        for (int it = 0; it < S; ++it)
            issue_rows_cp(it);
    } else if constexpr (STAGED) {
        if (tid == 0) {
            for (int i = 0; i < S; ++i)
                mbar_init(&sm_full[i], 1);
            mbar_init(&sm_never, 1);
            asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        }
        __syncthreads();
        if (warp == 0)
            for (int it = 0; it < S && it < n_it; ++it)
                issue_stage(it);
    } else {
        load_round(t0, kr0, vr0, ok0);
    }
    // register-streamed full layers: rounds 1 .. prefetch go to L2 now, later
    // rounds `prefetch` ahead of use
    auto row_at = [&](int t) { return t < t1 ? t : -1; };
    const int pf = (STAGED || SPARSE) ? 0 : a.prefetch;
    for (int d = 1; d <= pf; ++d)
        prefetch_round_l2(krows, vrows, t0 + d * step + warp * 8, lane, row_at);
    pdl_wait();

    // This lane's 8 dims of the group's G queries, as 4 dim pairs.
    float2 q2[G][4];
#pragma unroll
    for (int h = 0; h < G; ++h) {
        const uint4 qv = *reinterpret_cast<const uint4 *>(
            a.q + ((size_t)b * a.Hq + (size_t)g * G + h) * kHeadDim + c * 8);
        unpack8x2(qv, q2[h]);
    }

    const float c2 = a.scale * kLog2e;  // logits in log2 units for exp2
    float m[G], l[G];
    float2 o[G][4];  // un-normalised output, dim pairs
#pragma unroll
    for (int h = 0; h < G; ++h) {
        m[h] = -CUDART_INF_F;
        l[h] = 0.0f;
#pragma unroll
        for (int j = 0; j < 4; ++j)
            o[h][j] = make_float2(0.0f, 0.0f);
    }

    // One round: scores, online softmax and P V for this half-warp's U tokens.
    auto round = [&](int base, const uint4 (&kr)[U], const uint4 (&vr)[U], const bool (&ok)[U]) {
        const int tb = base + (warp * 2 + half) * U;  // this half-warp's first token

        // q . k over this lane's 8 dims (even and odd dims in the two
        // halves of a packed accumulator), then over the half-warp's 16
        // lanes, two (head, token) sums per packed add.
        static_assert(U % 2 == 0, "tokens are reduced in pairs");
        float2 dp[G][U / 2];  // (dot[h][2v], dot[h][2v+1])
#pragma unroll
        for (int u = 0; u < U; ++u) {
            float2 k2[4];
            unpack8x2(kr[u], k2);
#pragma unroll
            for (int h = 0; h < G; ++h) {
                float2 acc = __fmul2_rn(q2[h][0], k2[0]);
#pragma unroll
                for (int j = 1; j < 4; ++j)
                    acc = __ffma2_rn(q2[h][j], k2[j], acc);
                const float d = acc.x + acc.y;
                if (u & 1)
                    dp[h][u / 2].y = d;
                else
                    dp[h][u / 2].x = d;
            }
        }
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
            for (int v2 = 0; v2 < U / 2; ++v2)
#pragma unroll
                for (int off = 8; off >= 1; off >>= 1) {
                    const float2 t = make_float2(__shfl_xor_sync(kFull, dp[h][v2].x, off),
                                                 __shfl_xor_sync(kFull, dp[h][v2].y, off));
                    dp[h][v2] = __fadd2_rn(dp[h][v2], t);
                }
        float dot[G][U];
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
            for (int u = 0; u < U; ++u)
                dot[h][u] = (u & 1) ? dp[h][u / 2].y : dp[h][u / 2].x;

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
                const float2 al2 = make_float2(alpha, alpha);
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    o[h][j] = __fmul2_rn(o[h][j], al2);
                m[h] = m_new;
            } else {
#pragma unroll
                for (int u = 0; u < U; ++u)
                    p[h][u] = 0.0f;
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            float2 v2[4];
            unpack8x2(vr[u], v2);
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const float2 p2 = make_float2(p[h][u], p[h][u]);
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    o[h][j] = __ffma2_rn(p2, v2[j], o[h][j]);
            }
        }
    };
    if constexpr (STAGED == 1 && SPARSE) {
        const int slot0 = (warp * 2 + half) * U;
        const int trig = a.early_trigger > 0 ? max(n_it - a.early_trigger, 0) : -1;
        for (int it = 0; it < n_it; ++it) {
            if (it == trig)
                pdl_launch_dependents();
            cp_async_wait<S - 1>();  // this thread's copies of stage `it` have landed
            const unsigned char *kst = sm_stage + (it % S) * kStageBytes;
            const unsigned char *vst = kst + kStageBytes / 2;
            const int base = t0 + it * kTokPerRound;
            uint4 kr[U], vr[U];
            bool ok[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int t = base + slot0 + u;
                ok[u] = t < t1 && sm_rows[t - t0] >= 0;
                kr[u] = ok[u] ? lds128(kst + (slot0 + u) * kStageRowBytes + c * 16)
                              : make_uint4(0u, 0u, 0u, 0u);
                vr[u] = ok[u] ? lds128(vst + (slot0 + u) * kStageRowBytes + c * 16)
                              : make_uint4(0u, 0u, 0u, 0u);
            }
            round(base, kr, vr, ok);
            issue_rows_cp(it + S);  // refill the slot just consumed (its values are used above)
        }
        cp_async_wait<0>();
    } else if constexpr (STAGED) {
        int it = 0;
        bool failed = false;
        const uint64_t limit = a.wait_limit_us > 0 ? (uint64_t)a.wait_limit_us * 1000ull
                                                    : kWaitLimitNs;
        for (; it < n_it; ++it) {
            const int st = it % S;
            // false only if a copy did not complete within the limit:
            // reported, and the CTA's partial is discarded below
            const bool landed =
                (a.wait_test && it == 0) ? mbar_wait(&sm_never, 0u, limit)
                                         : mbar_wait(&sm_full[st], (unsigned)(it / S) & 1u, limit);
            const unsigned char *kst = sm_stage + st * kStageBytes;
            const unsigned char *vst = kst + kStageBytes / 2;
            const int base = t0 + it * kTokPerRound;
            const int slot0 = (warp * 2 + half) * U;
            uint4 kr[U], vr[U];
            bool ok[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int t = base + slot0 + u;
                ok[u] = t < t1 && (!SPARSE || sm_rows[t - t0] >= 0);
                kr[u] = ok[u] ? lds128(kst + (slot0 + u) * kStageRowBytes + c * 16)
                              : make_uint4(0u, 0u, 0u, 0u);
                vr[u] = ok[u] ? lds128(vst + (slot0 + u) * kStageRowBytes + c * 16)
                              : make_uint4(0u, 0u, 0u, 0u);
            }
            round(base, kr, vr, ok);
            failed = __syncthreads_or(!landed);  // also: every warp is done with stage st
            if (failed)
                break;
            if (warp == 0 && it + S < n_it) {
                // the ring slot is free: order the reads above before the async-proxy writes
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                issue_stage(it + S);
            }
        }
        if (failed) {
            // Every stage issued and not yet consumed (the one that did not
            // land, and those after it) lands before the CTA goes on: one
            // bounded wait each at the default limit, so no copy into this CTA's
            // shared memory is in flight when it exits.  Then the CTA takes
            // part in the split merge with an empty partial (m = -inf, l = 0),
            // so the (batch row, KV head)'s merge still runs and its ticket
            // returns to zero for the next launch on this workspace; the
            // output misses this split's tokens and the status word says so.
            if (tid == 0) {
                for (int j = it; j < n_it && j < it + S; ++j)
                    mbar_wait(&sm_full[j % S], (unsigned)(j / S) & 1u);
                atomicOr(a.status, kFlagWaitTimeout);
            }
            __syncthreads();
#pragma unroll
            for (int h = 0; h < G; ++h) {
                m[h] = -CUDART_INF_F;
                l[h] = 0.0f;
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    o[h][j] = make_float2(0.0f, 0.0f);
            }
        }
    } else {
        // rounds of this CTA: t0, t0 + step, ...; with early_trigger the next
        // kernel may launch from the start of round n_rounds - early_trigger
        const int n_rounds = t1 > t0 ? (t1 - t0 + step - 1) / step : 0;
        const int trig = a.early_trigger > 0 ? max(n_rounds - a.early_trigger, 0) : -1;
        if (trig == 0)
            pdl_launch_dependents();
        if (t0 < t1)
            round(t0, kr0, vr0, ok0);
        int ri = 1;
        for (int base = t0 + step; base < t1; base += step, ++ri) {
            uint4 kr[U], vr[U];
            bool ok[U];
            if (ri == trig)
                pdl_launch_dependents();
            if (pf > 0)
                prefetch_round_l2(krows, vrows, base + pf * step + warp * 8, lane, row_at);
            load_round(base, kr, vr, ok);
            round(base, kr, vr, ok);
        }
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
        for (int j = 0; j < 4; ++j) {
            const float2 oo = make_float2(__shfl_xor_sync(kFull, o[h][j].x, 16),
                                          __shfl_xor_sync(kFull, o[h][j].y, 16));
            o[h][j] = make_float2(o[h][j].x * sa + oo.x * so, o[h][j].y * sa + oo.y * so);
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
            dst[0] = make_float4(o[h][0].x, o[h][0].y, o[h][1].x, o[h][1].y);
            dst[1] = make_float4(o[h][2].x, o[h][2].y, o[h][3].x, o[h][3].y);
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
    finish_splits<G>(a, sm_o, sm_w, sm_M, sm_L, &sm_last, bg, split, nsplit_b, out_row0);
}

int g_carveout = -1;  // preferred shared-memory carveout (percent) for the attention kernels

template <int G, int STAGED>
constexpr size_t dyn_smem_bytes()
{
    return STAGED ? (size_t)staged_stages(G) * kStageBytes : 0;
}

// The dynamic shared-memory opt-in of the staged kernels, once per device.
template <int G, bool SPARSE, bool SELECT, bool CLUSTER, int STAGED>
cudaError_t configure_once()
{
    if (!STAGED)
        return cudaSuccess;
    static bool configured[64] = {false};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev >= 0 && dev < 64 && configured[dev])
        return cudaSuccess;
    e = cudaFuncSetAttribute(attention_kernel<G, SPARSE, SELECT, CLUSTER, STAGED>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)dyn_smem_bytes<G, STAGED>());
    if (e == cudaSuccess && dev >= 0 && dev < 64)
        configured[dev] = true;
    return e;
}

template <int G, bool SPARSE, bool SELECT, bool CLUSTER, int STAGED>
cudaError_t launch_one(const AttnArgs &a, int batch, bool pdl, cudaStream_t stream)
{
    auto kern = attention_kernel<G, SPARSE, SELECT, CLUSTER, STAGED>;
    if (g_carveout >= 0)
        cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, g_carveout);
    cudaError_t e0 = configure_once<G, SPARSE, SELECT, CLUSTER, STAGED>();
    if (e0 != cudaSuccess)
        return e0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)a.nsplit, (unsigned)a.Hkv, (unsigned)batch);
    cfg.blockDim = dim3(kAttnThreads);
    cfg.dynamicSmemBytes = dyn_smem_bytes<G, STAGED>();
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    int nattr = 1;
    if (CLUSTER) {
        if (a.nsplit > 8) {  // beyond the portable cluster size
            cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
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
    return cudaLaunchKernelEx(&cfg, kern, a);
}

template <int G, bool SPARSE, bool SELECT, int STAGED>
int occupancy_one()
{
    int n = 0;
    if (configure_once<G, SPARSE, SELECT, false, STAGED>() != cudaSuccess)
        return 1;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(
            &n, attention_kernel<G, SPARSE, SELECT, false, STAGED>, kAttnThreads,
            dyn_smem_bytes<G, STAGED>()) != cudaSuccess)
        return 1;
    return n > 0 ? n : 1;
}

// The cluster merge is built for the register-streamed kernels.
template <int G, bool SPARSE, bool SELECT>
cudaError_t launch_mode(bool cluster, int staged, const AttnArgs &a, int batch, bool pdl,
                        cudaStream_t st)
{
    if (cluster)
        return launch_one<G, SPARSE, SELECT, true, 0>(a, batch, pdl, st);
    if constexpr (SPARSE)
        if (staged == 2)
            return launch_one<G, SPARSE, SELECT, false, 2>(a, batch, pdl, st);
    return staged ? launch_one<G, SPARSE, SELECT, false, 1>(a, batch, pdl, st)
                  : launch_one<G, SPARSE, SELECT, false, 0>(a, batch, pdl, st);
}

template <int G>
cudaError_t launch_g(bool sparse, bool select, bool cluster, int staged, const AttnArgs &a,
                     int batch, bool pdl, cudaStream_t st)
{
    if (sparse)
        return launch_mode<G, true, false>(cluster, staged, a, batch, pdl, st);
    if (select)
        return launch_mode<G, false, true>(cluster, staged, a, batch, pdl, st);
    return launch_mode<G, false, false>(cluster, staged, a, batch, pdl, st);
}

}  // namespace

void set_attention_carveout(int percent) { g_carveout = percent; }

cudaError_t launch_attention(int G, bool sparse, bool select, bool cluster, int staged,
                             const AttnArgs &a, int batch, bool pdl, cudaStream_t stream)
{
    switch (G) {
    case 1:
        return launch_g<1>(sparse, select, cluster, staged, a, batch, pdl, stream);
    case 2:
        return launch_g<2>(sparse, select, cluster, staged, a, batch, pdl, stream);
    case 4:
        return launch_g<4>(sparse, select, cluster, staged, a, batch, pdl, stream);
    case 8:
        return launch_g<8>(sparse, select, cluster, staged, a, batch, pdl, stream);
    default:
        return cudaErrorInvalidValue;
    }
}

int attention_ctas_per_sm(int G, bool sparse, bool select, int staged)
{
#define TD_OCC_G(GG)                                                                      \
    case GG:                                                                              \
        if (sparse)                                                                       \
            return staged == 2 ? occupancy_one<GG, true, false, 2>()                      \
                               : (staged ? occupancy_one<GG, true, false, 1>()            \
                                         : occupancy_one<GG, true, false, 0>());          \
        if (select)                                                                       \
            return staged ? occupancy_one<GG, false, true, 1>()                           \
                          : occupancy_one<GG, false, true, 0>();                          \
        return staged ? occupancy_one<GG, false, false, 1>()                              \
                      : occupancy_one<GG, false, false, 0>();
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
