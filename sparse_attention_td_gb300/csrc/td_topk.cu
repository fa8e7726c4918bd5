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
// Method: exact radix select on order-preserving 32-bit keys, one CTA (1024
// or 512 threads) per row:
//   1. an 11-bit histogram of the keys' top bits picks the bin holding the
//      k-th largest key.  In a selection layer the attention kernel that
//      wrote the scores already built it (and this kernel clears it again);
//      for caller-given scores it is counted here.
//   2. One read of the row: keys above that bin are marked in a shared-memory
//      bitmap of the row's positions, and the bin's (key, position) pairs
//      are gathered into shared memory.  The select finishes on the gathered
//      pairs (in one warp when there are few): the k-th key T and, when only
//      some keys equal to T fit in the set, the largest position P that still
//      does (the lowest positions win ties).  The selected pairs are marked.
//   3. The set is written in position order by a block-wide scan of the
//      bitmap.
// Loads are batched sixteen scores per thread (four float4 loads on 16-byte
// aligned rows).  Rows longer than the bitmap, or a
// threshold bin larger than the shared-memory buffer (heavily tied scores),
// fall back to streaming passes and an ordered compaction of the row.
#include <cooperative_groups.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "td_attn_common.cuh"  // order_key (the attention kernels' first-digit
                               // histogram bins scores with the same key),
                               // launch-dependency waits
#include "td_internal.h"

namespace td {
namespace {

constexpr int kBatch = 16;              // loads in flight per thread
constexpr int kBatchV = 4;              // float4 loads in flight per thread (16 scores)
// Threshold bins up to this size finish in one warp (no block barriers);
// larger ones take block-wide radix passes.  Measured on GB300: 256 beats
// 2048 by 1-4 us per selection layer on 10K-32K rows, whose bins hold
// several hundred to ~2000 pairs (one warp makes a serial pass per 32).
constexpr unsigned kWarpSelectMax = 256;
constexpr int kBits1 = kSelectBits;     // first digit: key bits 31..21
constexpr int kBins1 = kSelectBins;     // 2048
constexpr int kBitmapWords = kTopkBitmapBits / 32;
constexpr int kSubHists = 4;            // pass-1 sub-histograms (less atomic contention)

// Programmatic dependent launch: the scores come from the kernel just before
// this one, so the kernel waits for it (pdl_wait); the next layer's kernel may
// launch right away (it waits for this one before reading the index set).

// The kernel is instantiated for two block sizes: 1024 threads (one CTA per
// SM, for launches with fewer rows than SMs) and 512 threads (two CTAs per SM
// in 64 registers a thread, so many rows run in a single wave).
template <int NT>
struct TopkCfg {
    static constexpr int kT = NT;
    static constexpr int kWarps = NT / 32;
    static constexpr int kWordsPerThread = kBitmapWords / NT;
    static constexpr int kCand = NT >= 1024 ? kTopkCandidates : kTopkCandidates / 2;  // (key, pos) pairs
    static constexpr int kMinBlocks = 1024 / NT;
};

constexpr int kShortList = 256;         // pairs one warp finishes after the second digit

template <int NT>
struct TopkSmem {
    static constexpr int kWarps = NT / 32;
    unsigned hist[kBins1];              // first-digit histogram, later a 256-bin scratch histogram
    unsigned hist2[256];                // second digit (key bits 20..13) of the threshold bin's pairs
    unsigned scan[32];                  // per-warp partial sums (entries >= kWarps stay unused)
    unsigned tot[kBatch * kWarps];
    unsigned pre[kBatch * kWarps];
    unsigned res[2];                    // digit, remaining rank
    unsigned cand_count;
    unsigned cut[2];                    // the k-th key T and the largest kept position P
    unsigned short_count;               // pairs of the narrowed threshold bin
    uint32_t short_key[kShortList];     // the narrowed bin's pairs (bin_cut)
    int32_t short_pos[kShortList];
    unsigned slice_total;               // cluster path: positions this CTA's slice keeps
    unsigned bitmap[kBitmapWords];      // selected positions of rows up to kTopkBitmapBits long
};

// Block-wide search over a histogram of NB bins (digit = bin index): the
// digit d with count(> d) < r <= count(>= d).  Writes d and r - count(> d)
// to sm.res.  All threads must call it.
template <int NB, int NT>
__device__ void find_digit(TopkSmem<NT> &sm, const unsigned *hist, unsigned r)
{
    constexpr int kT = NT, kWarps = NT / 32;
    constexpr int per = NB >= kT ? NB / kT : 1;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int first = NB - 1 - tid * per;  // this thread's highest bin
    unsigned c = 0;
    if (first >= 0)
        for (int i = 0; i < per; ++i)
            c += hist[first - i];
    unsigned incl = c;
    for (int off = 1; off < 32; off <<= 1) {
        const unsigned v = __shfl_up_sync(kFull, incl, off);
        if (lane >= off)
            incl += v;
    }
    if (lane == 31)
        sm.scan[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        unsigned w = lane < kWarps ? sm.scan[lane] : 0u, wi = w;
        for (int off = 1; off < 32; off <<= 1) {
            const unsigned v = __shfl_up_sync(kFull, wi, off);
            if (lane >= off)
                wi += v;
        }
        sm.scan[lane] = wi - w;  // exclusive offset of each warp
    }
    __syncthreads();
    incl += sm.scan[warp];
    const unsigned excl = incl - c;
    if (c > 0 && excl < r && r <= incl) {
        unsigned run = excl;
        for (int i = 0; i < per; ++i) {
            const unsigned h = hist[first - i];
            if (run + h >= r) {
                sm.res[0] = (unsigned)(first - i);
                sm.res[1] = r - run;
                break;
            }
            run += h;
        }
    }
    __syncthreads();
}

// Exclusive prefix sum of v over the block (thread order); *total gets the sum.
template <int NT>
__device__ __forceinline__ unsigned block_exclusive_sum(TopkSmem<NT> &sm, unsigned v, unsigned *total)
{
    constexpr int kWarps = NT / 32;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    unsigned incl = v;
    for (int off = 1; off < 32; off <<= 1) {
        const unsigned t = __shfl_up_sync(kFull, incl, off);
        if (lane >= off)
            incl += t;
    }
    if (lane == 31)
        sm.scan[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const unsigned w = lane < kWarps ? sm.scan[lane] : 0u;
        unsigned wi = w;
        for (int off = 1; off < 32; off <<= 1) {
            const unsigned t = __shfl_up_sync(kFull, wi, off);
            if (lane >= off)
                wi += t;
        }
        sm.scan[lane] = wi - w;
        if (lane == 31)
            sm.res[0] = wi;
    }
    __syncthreads();
    const unsigned excl = incl - v + sm.scan[warp];
    *total = sm.res[0];
    __syncthreads();
    return excl;
}

// Calls f(key, pos) for every position of the row, kBatch loads in flight per thread.
template <int NT, class F>
__device__ __forceinline__ void stream_row(const float *s, int n, F f)
{
    constexpr int kT = NT;
    for (int base = 0; base < n; base += kT * kBatch) {
        float v[kBatch];
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
            const int i = base + j * kT + (int)threadIdx.x;
            v[j] = i < n ? __ldcg(&s[i]) : 0.0f;
        }
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
            const int i = base + j * kT + (int)threadIdx.x;
            if (i < n)
                f(order_key(v[j]), i);
        }
    }
}

// Radix select over a stream of (value, item) pairs that pass `keep`: the
// r-th largest value among them, digits of 8 bits over bits [hi_bit..0],
// starting from `prefix`/`mask` (bits already fixed).  `src(f)` must call f
// for every pair.  Returns the value; *rank_out receives r minus the count of
// larger values (how many items equal to the result belong in the set) and
// *eq_out the number of items equal to it.
template <int NT, class Src>
__device__ uint32_t radix_select(TopkSmem<NT> &sm, Src src, int hi_bit, uint32_t prefix,
                                 uint32_t mask, unsigned r, unsigned *rank_out, unsigned *eq_out)
{
    unsigned *hist = sm.hist;
    unsigned last_count = 0;
    for (int top = hi_bit; top >= 0; top -= 8) {
        const int width = top + 1 < 8 ? top + 1 : 8;
        const int shift = top + 1 - width;
        const unsigned dmask = (1u << width) - 1u;
        for (int i = threadIdx.x; i < 256; i += NT)
            hist[i] = 0u;
        __syncthreads();
        src([&](uint32_t val, int) {
            if ((val & mask) == prefix)
                atomicAdd(&hist[(val >> shift) & dmask], 1u);
        });
        __syncthreads();
        find_digit<256>(sm, hist, r);
        const unsigned d = sm.res[0];
        r = sm.res[1];
        last_count = hist[d];
        prefix |= d << shift;
        mask |= dmask << shift;
        __syncthreads();
    }
    *rank_out = r;
    *eq_out = last_count;
    return prefix;
}

// One warp's search of a 256-bin histogram, lane L holding bins 255 - 8L down
// to 248 - 8L: the digit d with count(> d) < r <= count(>= d).  Returns d to
// every lane; *rank_out = r - count(> d), *cnt_out = count(d).
__device__ __forceinline__ uint32_t warp_find_digit(const unsigned *hist, unsigned r,
                                                    unsigned *rank_out, unsigned *cnt_out)
{
    const int lane = threadIdx.x & 31;
    unsigned mine = 0;
    for (int i = 0; i < 8; ++i)
        mine += hist[255 - 8 * lane - i];
    unsigned incl = mine;
    for (int off = 1; off < 32; off <<= 1) {
        const unsigned t = __shfl_up_sync(kFull, incl, off);
        if (lane >= off)
            incl += t;
    }
    const unsigned excl = incl - mine;
    const bool owner = excl < r && r <= incl;
    unsigned d = 0, rn = 0, cnt = 0;
    if (owner) {
        unsigned run = excl;
        for (int i = 0; i < 8; ++i) {
            const unsigned bin = 255 - 8 * lane - i;
            const unsigned h = hist[bin];
            if (run + h >= r) {
                d = bin;
                rn = r - run;
                cnt = h;
                break;
            }
            run += h;
        }
    }
    const int src = __ffs(__ballot_sync(kFull, owner)) - 1;
    *rank_out = __shfl_sync(kFull, rn, src);
    *cnt_out = __shfl_sync(kFull, cnt, src);
    return __shfl_sync(kFull, d, src);
}

// One warp's radix select over n items of a shared-memory list: the r-th
// largest value val(i) among the items with keep(i), digits of 8 bits over
// bits [hi_bit..0] below the already fixed `prefix`/`mask`.  `hist` is a
// 256-bin scratch histogram private to the warp.  Returns the value;
// *rank_out = how many items equal to it belong in the set, *eq_out = how
// many items equal it.  Warp-synchronous: no block barrier.
template <class ValF, class KeepF>
__device__ uint32_t warp_select(unsigned *hist, unsigned n, ValF val, KeepF keep, int hi_bit,
                                uint32_t prefix, uint32_t mask, unsigned r, unsigned *rank_out,
                                unsigned *eq_out)
{
    const int lane = threadIdx.x & 31;
    unsigned last = 0;
    for (int top = hi_bit; top >= 0; top -= 8) {
        const int width = top + 1 < 8 ? top + 1 : 8;
        const int shift = top + 1 - width;
        const unsigned dmask = (1u << width) - 1u;
        for (int i = lane; i < 256; i += 32)
            hist[i] = 0u;
        __syncwarp();
        for (unsigned i = lane; i < n; i += 32) {
            if (!keep(i))
                continue;
            const uint32_t v = val(i);
            if ((v & mask) == prefix)
                atomicAdd(&hist[(v >> shift) & dmask], 1u);
        }
        __syncwarp();
        unsigned rn;
        const uint32_t d = warp_find_digit(hist, r, &rn, &last);
        r = rn;
        prefix |= d << shift;
        mask |= dmask << shift;
        __syncwarp();
    }
    *rank_out = r;
    *eq_out = last;
    return prefix;
}

// The cut of a threshold bin whose cnt (key, position) pairs are in shared
// memory (keys share prefix1 under mask1): T = the r1-th largest key, P = the
// largest position kept among keys equal to T (lower positions win ties;
// INT_MAX when every key equal to T is kept).  A bin of up to warp_max pairs
// is finished by one warp.  A larger one is narrowed first by its pairs' next
// 8-bit digit (key bits 20..13), whose counts the caller's row pass left in
// sm.hist2 (visible to every thread on entry): every warp finds
// the digit holding the r1-th key, the block copies that digit's pairs (a
// few, unless the keys are heavily tied) to a short list, and one warp
// finishes there; a digit with more than kShortList pairs takes block-wide
// radix passes over the bin.  sm.short_count is zero on entry.  All threads
// call it; the cut is in sm.cut on return.
template <int NT>
__device__ void bin_cut(TopkSmem<NT> &sm, const uint32_t *cand_key, const int32_t *cand_pos,
                        unsigned cnt, uint32_t prefix1, uint32_t mask1, unsigned r1,
                        unsigned warp_max)
{
    constexpr int kT = NT;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (cnt <= warp_max) {
        if (warp == 0) {
            unsigned need, neq;
            const uint32_t t = warp_select(
                sm.hist, cnt, [&](unsigned i) { return cand_key[i]; },
                [&](unsigned) { return true; }, 31 - kBits1, prefix1, mask1, r1, &need, &neq);
            int p_cut = 0x7fffffff;
            if (need < neq) {
                unsigned r2, e2;
                p_cut = (int)~warp_select(
                    sm.hist, cnt, [&](unsigned i) { return ~(uint32_t)cand_pos[i]; },
                    [&](unsigned i) { return cand_key[i] == t; }, 31, 0u, 0u, need, &r2, &e2);
            }
            if (lane == 0) {
                sm.cut[0] = t;
                sm.cut[1] = (unsigned)p_cut;
            }
        }
        __syncthreads();
        return;
    }
    // second digit: key bits 20..13
    constexpr int kShift2 = 32 - kBits1 - 8;
    // every warp finds the digit holding the r1-th key (no block barrier)
    unsigned r2, n2;
    const uint32_t d2 = warp_find_digit(sm.hist2, r1, &r2, &n2);
    const uint32_t prefix2 = prefix1 | (d2 << kShift2);
    const uint32_t mask2 = mask1 | (0xffu << kShift2);
    if (n2 <= (unsigned)kShortList) {
        for (unsigned i = tid; i < cnt; i += kT)
            if ((cand_key[i] & mask2) == prefix2) {
                const unsigned slot = atomicAdd(&sm.short_count, 1u);  // n2 slots in all
                sm.short_key[slot] = cand_key[i];
                sm.short_pos[slot] = cand_pos[i];
            }
        __syncthreads();
        if (warp == 0) {
            unsigned need, neq;
            const uint32_t t = warp_select(
                sm.hist, n2, [&](unsigned i) { return sm.short_key[i]; },
                [&](unsigned) { return true; }, kShift2 - 1, prefix2, mask2, r2, &need, &neq);
            int p_cut = 0x7fffffff;
            if (need < neq) {
                unsigned rr, ee;
                p_cut = (int)~warp_select(
                    sm.hist, n2, [&](unsigned i) { return ~(uint32_t)sm.short_pos[i]; },
                    [&](unsigned i) { return sm.short_key[i] == t; }, 31, 0u, 0u, need, &rr, &ee);
            }
            if (lane == 0) {
                sm.cut[0] = t;
                sm.cut[1] = (unsigned)p_cut;
            }
        }
        __syncthreads();
        return;
    }
    // heavily tied: block-wide radix passes over the bin's remaining digits
    auto cand_src = [&](auto f) {
        for (unsigned i = tid; i < cnt; i += kT)
            f(cand_key[i], cand_pos[i]);
    };
    unsigned need_eq, n_eq;
    const uint32_t T = radix_select(sm, cand_src, kShift2 - 1, prefix2, mask2, r2, &need_eq, &n_eq);
    int P = 0x7fffffff;
    if (need_eq < n_eq) {
        auto eq_src = [&](auto f) {
            for (unsigned i = tid; i < cnt; i += kT)
                if (cand_key[i] == T)
                    f(~(uint32_t)cand_pos[i], 0);
        };
        unsigned r_dummy, e_dummy;
        P = (int)~radix_select(sm, eq_src, 31, 0u, 0u, need_eq, &r_dummy, &e_dummy);
    }
    if (tid == 0) {
        sm.cut[0] = T;
        sm.cut[1] = (unsigned)P;
    }
    __syncthreads();
}

// Row length n of batch row b (clamped to [0, Nmax]; out-of-range lengths
// are flagged once per batch row by `flag`).
__device__ __forceinline__ int topk_row_len(const TopkArgs &a, int b, bool flag)
{
    int n = a.seq_lens[b];
    if (n < 0 || n > a.Nmax) {
        if (flag)
            atomicOr(a.status, kFlagSeqLenOutOfRange);
        n = n < 0 ? 0 : a.Nmax;
    }
    return n;
}

// Positions to select in row bg: top_k, or the row's budget (at most top_k).
__device__ __forceinline__ int topk_row_budget(const TopkArgs &a, size_t bg)
{
    int k = a.top_k;
    if (a.row_k) {
        const int rk = __ldcg(a.row_k + bg);
        k = rk < 0 ? 0 : (rk < a.top_k ? rk : a.top_k);
    }
    return k;
}

// The whole selection of row (b, KV head g) by one CTA of NT threads, with
// the dynamic shared memory of topk_kernel<NT>.  Called after the wait for
// the kernel that wrote the scores.  Not inlined: the clustered kernel calls
// it only for the rows it cannot take, and keeping its code out of that
// kernel's body keeps the common path small.
template <int NT>
__device__ __noinline__ void topk_row(const TopkArgs &a, int g, int b, unsigned char *smem_raw)
{
    using C = TopkCfg<NT>;
    constexpr int kT = C::kT, kWarps = C::kWarps, kWordsPerThread = C::kWordsPerThread;
    TopkSmem<NT> &sm = *reinterpret_cast<TopkSmem<NT> *>(smem_raw);
    uint32_t *cand_key = reinterpret_cast<uint32_t *>(smem_raw + sizeof(TopkSmem<NT>));
    int32_t *cand_pos = reinterpret_cast<int32_t *>(cand_key + C::kCand);

    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    const size_t bg = (size_t)b * a.Hkv + g;
    const int kcap = a.top_k;  // row length of the output
    const int n = topk_row_len(a, b, tid == 0 && g == 0);
    const float *s = a.scores + bg * (size_t)a.Nmax;
    int32_t *out = a.idx + bg * (size_t)kcap;
    const int k = topk_row_budget(a, bg);  // positions to select in this row
    if (a.counts && tid == 0)
        a.counts[bg] = k < n ? k : n;

    unsigned *ghist = a.hist ? a.hist + bg * kBins1 : nullptr;
    if (n <= k || k == 0) {  // every position is kept, or none
        for (int j = tid; j < kcap; j += kT)
            out[j] = (j < n && j < k) ? j : -1;
        if (ghist)
            for (int i = tid; i < kBins1; i += kT)
                ghist[i] = 0u;  // leave the fused histogram zero for the next selection
        return;
    }

    const int vec_n = (((uintptr_t)s & 15u) == 0) ? n / 4 : 0;  // whole float4 groups
    const bool use_bitmap = n <= kTopkBitmapBits;
    // The first batch of the row's float4 groups, requested before the
    // first-digit search it waits for (the row pass below starts with it).
    float4 v[kBatchV];
    auto load_batch = [&](int base) {
#pragma unroll
        for (int j = 0; j < kBatchV; ++j) {
            const int i4 = base + j * kT + tid;
            v[j] = i4 < vec_n ? __ldcg(reinterpret_cast<const float4 *>(s) + i4)
                              : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        }
    };

    // 1. histogram of the top 11 bits: from the attention kernel that wrote
    //    the scores (then cleared for the next selection), else counted here
    if (tid == 0) {
        sm.cand_count = 0u;
        sm.short_count = 0u;
    }
    if (ghist) {
        load_batch(0);
        for (int i = tid; i < kBins1; i += kT) {
            sm.hist[i] = __ldcg(&ghist[i]);
            ghist[i] = 0u;
        }
    } else {
        // sub-histograms (less atomic contention) in the candidate area, unused until pass 2
        unsigned *sub = reinterpret_cast<unsigned *>(cand_key);
        for (int i = tid; i < kSubHists * kBins1; i += kT)
            sub[i] = 0u;
        __syncthreads();
        unsigned *mine = sub + (warp % kSubHists) * kBins1;
        stream_row<NT>(s, n, [&](uint32_t key, int) { atomicAdd(&mine[key >> (32 - kBits1)], 1u); });
        __syncthreads();
        for (int i = tid; i < kBins1; i += kT) {
            unsigned t = 0;
            for (int h = 0; h < kSubHists; ++h)
                t += sub[h * kBins1 + i];
            sm.hist[i] = t;
        }
        load_batch(0);
    }
    // the bitmap and the second-digit counts start empty
    if (use_bitmap)
        for (int w = tid; w < (n + 31) / 32; w += kT)
            sm.bitmap[w] = 0u;
    for (int i = tid; i < 256; i += kT)
        sm.hist2[i] = 0u;
    __syncthreads();
    find_digit<kBins1>(sm, sm.hist, (unsigned)k);
    const uint32_t d1 = sm.res[0];
    const unsigned r1 = sm.res[1];
    const unsigned bin_count = sm.hist[d1];
    __syncthreads();

    const uint32_t prefix1 = d1 << (32 - kBits1);
    const uint32_t mask1 = ~0u << (32 - kBits1);
    uint32_t T;
    unsigned need_eq, n_eq;
    int P = 0x7fffffff;  // largest kept position among keys == T
    constexpr int kShift2 = 32 - kBits1 - 8;  // second digit: key bits 20..13
    if (bin_count <= (unsigned)C::kCand) {
        // 2. gather the threshold bin into shared memory, finish there; rows
        //    that fit the bitmap also mark every key above the bin as selected
        const uint32_t top_of_bin = prefix1 | ~mask1;  // largest key inside the threshold bin
        // Aligned rows: a thread takes 4 consecutive scores per load, so a warp
        // covers 128 positions = 4 bitmap words (a word's 8 nibbles are OR-ed
        // together with 3 shuffles).  A key is in the threshold bin (above it)
        // when its first digit equals (exceeds) d1.  The bin holds a few
        // percent of the row at most, so each hit takes its candidate slot
        // with its own shared-memory atomic (no per-group warp scan) and
        // counts its second digit.
        for (int base = 0; base < vec_n; base += kT * kBatchV) {
            if (base > 0)
                load_batch(base);
#pragma unroll
            for (int j = 0; j < kBatchV; ++j) {
                const int i4 = base + j * kT + tid;
                const int pos0 = 4 * i4;
                const bool live = i4 < vec_n;
                const float f[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
                uint32_t key[4];
                unsigned hitm = 0u, abovem = 0u;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    key[e] = order_key(f[e]);
                    const uint32_t dg = key[e] >> (32 - kBits1);
                    hitm |= (live && dg == d1) ? (1u << e) : 0u;
                    abovem |= (live && dg > d1) ? (1u << e) : 0u;
                }
                if (use_bitmap) {
                    unsigned word = abovem << (4 * (lane & 7));
                    word |= __shfl_xor_sync(kFull, word, 1);
                    word |= __shfl_xor_sync(kFull, word, 2);
                    word |= __shfl_xor_sync(kFull, word, 4);
                    if ((lane & 7) == 0 && live)
                        sm.bitmap[pos0 >> 5] = word;
                }
                if (hitm) {  // at most bin_count <= kCand hits in all: slots stay in range
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        if (hitm & (1u << e)) {
                            const unsigned slot = atomicAdd(&sm.cand_count, 1u);
                            cand_key[slot] = key[e];
                            cand_pos[slot] = pos0 + e;
                            atomicAdd(&sm.hist2[(key[e] >> kShift2) & 0xffu], 1u);
                        }
                }
            }
        }
        __syncthreads();  // whole-word bitmap stores above land before the tail ORs into a word
        // the rest (unaligned rows, or the tail after the last whole group), one score per thread
        for (int base = 4 * vec_n; base < n; base += kT * kBatch) {
            float v[kBatch];
#pragma unroll
            for (int j = 0; j < kBatch; ++j) {
                const int i = base + j * kT + tid;
                v[j] = i < n ? __ldcg(&s[i]) : 0.0f;
            }
#pragma unroll
            for (int j = 0; j < kBatch; ++j) {
                const int i = base + j * kT + tid;
                const uint32_t key = order_key(v[j]);
                const bool hit = i < n && (key & mask1) == prefix1;
                if (use_bitmap && i < n && key > top_of_bin)  // may share a word with the vector part
                    atomicOr(&sm.bitmap[i >> 5], 1u << (i & 31));
                const unsigned m = __ballot_sync(kFull, hit);
                if (m) {  // warp-uniform
                    unsigned slot0 = 0;
                    if (lane == 0)
                        slot0 = atomicAdd(&sm.cand_count, (unsigned)__popc(m));
                    slot0 = __shfl_sync(kFull, slot0, 0);
                    if (hit) {
                        const unsigned slot = slot0 + __popc(m & ((1u << lane) - 1u));
                        cand_key[slot] = key;
                        cand_pos[slot] = i;
                        atomicAdd(&sm.hist2[(key >> kShift2) & 0xffu], 1u);
                    }
                }
            }
        }
        __syncthreads();
        const unsigned cnt = sm.cand_count;
        const unsigned warp_max = a.warp_select_max > 0 ? (unsigned)a.warp_select_max : kWarpSelectMax;
        bin_cut<NT>(sm, cand_key, cand_pos, cnt, prefix1, mask1, r1, warp_max);
        T = sm.cut[0];
        P = (int)sm.cut[1];
        if (use_bitmap) {
            // mark the selected part of the threshold bin
            for (unsigned i = tid; i < cnt; i += kT) {
                const uint32_t key = cand_key[i];
                const int pos = cand_pos[i];
                if (key > T || (key == T && pos <= P))
                    atomicOr(&sm.bitmap[pos >> 5], 1u << (pos & 31));
            }
            __syncthreads();
        }
        if (use_bitmap) {
            // write the set in position order by scanning the bitmap (no second
            // row read); the row's words are spread evenly over the threads
            const int words = (n + 31) / 32;
            const int wpt = (words + kT - 1) / kT;  // <= kWordsPerThread
            const int w0 = tid * wpt;
            unsigned w[kWordsPerThread];
            unsigned count = 0;
#pragma unroll
            for (int j = 0; j < kWordsPerThread; ++j) {
                const int wi = w0 + j;
                w[j] = (j < wpt && wi < words) ? sm.bitmap[wi] : 0u;
                count += __popc(w[j]);
            }
            unsigned total;
            unsigned slot = block_exclusive_sum(sm, count, &total);
#pragma unroll
            for (int j = 0; j < kWordsPerThread; ++j) {
                unsigned word = w[j];
                while (word) {
                    const int bit = __ffs(word) - 1;
                    word &= word - 1u;
                    if (slot < (unsigned)k)  // exactly k bits are set; the bound only guards memory
                        out[slot] = (w0 + j) * 32 + bit;
                    ++slot;
                }
            }
            for (int j = k + tid; j < kcap; j += kT)
                out[j] = -1;  // a per-row budget below the row length
            return;
        }
    } else {
        // threshold bin too large for shared memory: stream the remaining digits
        auto row_src = [&](auto f) { stream_row<NT>(s, n, f); };
        T = radix_select(sm, row_src, 31 - kBits1, prefix1, mask1, r1, &need_eq, &n_eq);
        if (need_eq < n_eq) {
            auto eq_src = [&](auto f) {
                stream_row<NT>(s, n, [&](uint32_t key, int i) {
                    if (key == T)
                        f(~(uint32_t)i, 0);
                });
            };
            unsigned r_dummy, e_dummy;
            P = (int)~radix_select(sm, eq_src, 31, 0u, 0u, need_eq, &r_dummy, &e_dummy);
        }
    }
    __syncthreads();

    // 3. ordered compaction: keys > T, and keys == T at positions <= P
    unsigned out_base = 0;
    for (int base = 0; base < n; base += kT * kBatch) {
        float v[kBatch];
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
            const int i = base + j * kT + tid;
            v[j] = i < n ? __ldcg(&s[i]) : 0.0f;
        }
        unsigned bal[kBatch];
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
            const int i = base + j * kT + tid;
            const uint32_t key = order_key(v[j]);
            const bool take = i < n && (key > T || (key == T && i <= P));
            bal[j] = __ballot_sync(kFull, take);
            if (lane == 0)
                sm.tot[j * kWarps + warp] = __popc(bal[j]);
        }
        __syncthreads();
        if (warp == 0) {
            // exclusive scan of the 256 counts in (j, warp) order = position order
            constexpr int per = kBatch * kWarps / 32;  // counts per lane, position order
            unsigned c[per], sum = 0;
#pragma unroll
            for (int e = 0; e < per; ++e) {
                c[e] = sm.tot[lane * per + e];
                sum += c[e];
            }
            unsigned incl = sum;
            for (int off = 1; off < 32; off <<= 1) {
                const unsigned t = __shfl_up_sync(kFull, incl, off);
                if (lane >= off)
                    incl += t;
            }
            unsigned run = incl - sum;
#pragma unroll
            for (int e = 0; e < per; ++e) {
                sm.pre[lane * per + e] = run;
                run += c[e];
            }
            if (lane == 31)
                sm.res[0] = incl;  // super-tile total
        }
        __syncthreads();
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
            if (bal[j] & (1u << lane)) {
                const unsigned slot = out_base + sm.pre[j * kWarps + warp] +
                                      __popc(bal[j] & ((1u << lane) - 1u));
                if (slot < (unsigned)k)  // exactly k are taken; the bound only guards memory
                    out[slot] = base + j * kT + tid;
            }
        }
        out_base += sm.res[0];
        __syncthreads();
    }
    for (int j = k + tid; j < kcap; j += kT)
        out[j] = -1;  // a per-row budget below the row length
}

// One CTA per row (grid: KV heads x batch rows).
template <int NT>
__global__ void __launch_bounds__(NT, TopkCfg<NT>::kMinBlocks)
topk_kernel(const TopkArgs a)
{
    extern __shared__ __align__(16) unsigned char smem_raw[];
    pdl_wait();
    pdl_launch_dependents();
    topk_row<NT>(a, blockIdx.x, blockIdx.y, smem_raw);
}

namespace cg = cooperative_groups;
constexpr int kClusterNT = 1024;  // threads of each CTA of a row's cluster

// A cluster of CS CTAs per row (grid: CS x KV heads x batch rows), for
// launches with few, long rows, where one CTA per row would leave most SMs
// idle.  Rank r takes the positions [r * L, (r + 1) * L) of the row (L a
// multiple of 128): it marks the keys above the threshold bin in its slice of
// the position bitmap (its own shared memory) and gathers the bin's (key,
// position) pairs.  Rank 0 copies every rank's pairs through distributed
// shared memory, finishes the select (T, P) as topk_row does, and every rank
// reads the cut back, marks its selected pairs, and writes its slice of the
// set after the counts of the slices before it.  The result is the same set,
// in the same order, as topk_row.  Without the attention kernel's first-digit
// histogram each rank counts its slice's and the ranks sum them.  A row whose
// threshold bin exceeds the candidate buffer, a row longer than the bitmap,
// or a row that keeps every position (or none), is done by rank 0 alone with
// topk_row.
template <int CS>
__global__ void __cluster_dims__(CS, 1, 1) __launch_bounds__(kClusterNT, 1)
topk_cluster_kernel(const TopkArgs a)
{
    constexpr int NT = kClusterNT;
    using C = TopkCfg<NT>;
    constexpr int kT = C::kT;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    TopkSmem<NT> &sm = *reinterpret_cast<TopkSmem<NT> *>(smem_raw);
    uint32_t *cand_key = reinterpret_cast<uint32_t *>(smem_raw + sizeof(TopkSmem<NT>));
    int32_t *cand_pos = reinterpret_cast<int32_t *>(cand_key + C::kCand);
    cg::cluster_group cluster = cg::this_cluster();
    const int rank = (int)cluster.block_rank();
    const int g = blockIdx.y, b = blockIdx.z, tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    const size_t bg = (size_t)b * a.Hkv + g;

    pdl_wait();
    pdl_launch_dependents();
    const int n = topk_row_len(a, b, rank == 0 && tid == 0 && g == 0);
    const int k = topk_row_budget(a, bg);
    if (n <= k || k == 0 || n > kTopkBitmapBits) {
        if (rank == 0)
            topk_row<NT>(a, g, b, smem_raw);
        return;  // no rank touched another's shared memory
    }
    // this rank's slice of the row
    const int L = ((n + CS - 1) / CS + 127) / 128 * 128;
    const int lo = rank * L;
    const int hi = min(n, lo + L);
    const int len = hi > lo ? hi - lo : 0;
    const float *s = a.scores + bg * (size_t)a.Nmax + lo;

    unsigned *ghist = a.hist ? a.hist + bg * kBins1 : nullptr;
    if (ghist) {
        for (int i = tid; i < kBins1; i += kT)
            sm.hist[i] = __ldcg(&ghist[i]);
    } else {
        // the slice's first-digit counts (sub-histograms in the candidate
        // area), then the row's: every rank sums all ranks' counts
        unsigned *sub = reinterpret_cast<unsigned *>(cand_key);
        for (int i = tid; i < kSubHists * kBins1; i += kT)
            sub[i] = 0u;
        __syncthreads();
        unsigned *mine = sub + (warp % kSubHists) * kBins1;
        for (int base = 0; base < len; base += kT * kBatch) {
            float v[kBatch];
#pragma unroll
            for (int j = 0; j < kBatch; ++j) {
                const int i = base + j * kT + tid;
                v[j] = i < len ? __ldcg(&s[i]) : 0.0f;
            }
#pragma unroll
            for (int j = 0; j < kBatch; ++j)
                if (base + j * kT + tid < len)
                    atomicAdd(&mine[order_key(v[j]) >> (32 - kBits1)], 1u);
        }
        __syncthreads();
        for (int i = tid; i < kBins1; i += kT) {
            unsigned t = 0;
            for (int h = 0; h < kSubHists; ++h)
                t += sub[h * kBins1 + i];
            sm.hist[i] = t;
        }
        cluster.sync();  // every rank's slice counts are in its sm.hist
        unsigned *row_hist = sub;  // the sub-histograms are no longer needed
        for (int i = tid; i < kBins1; i += kT) {
            unsigned t = 0;
            for (int rr = 0; rr < CS; ++rr)
                t += *cluster.map_shared_rank(&sm.hist[i], rr);
            row_hist[i] = t;
        }
        cluster.sync();  // nobody still reads another rank's slice counts
        for (int i = tid; i < kBins1; i += kT)
            sm.hist[i] = row_hist[i];
    }
    if (tid == 0) {
        sm.cand_count = 0u;
        sm.short_count = 0u;
    }
    __syncthreads();
    find_digit<kBins1>(sm, sm.hist, (unsigned)k);
    const uint32_t d1 = sm.res[0];
    const unsigned r1 = sm.res[1];
    const unsigned bin_count = sm.hist[d1];
    __syncthreads();
    cluster.sync();  // every rank has read the histogram
    if (bin_count > (unsigned)C::kCand) {
        if (rank == 0)
            topk_row<NT>(a, g, b, smem_raw);  // reads the histogram again and clears it
        return;
    }
    if (rank == 0 && ghist)
        for (int i = tid; i < kBins1; i += kT)
            ghist[i] = 0u;  // leave the fused histogram zero for the next selection

    for (int w = tid; w < (len + 31) / 32; w += kT)
        sm.bitmap[w] = 0u;
    for (int i = tid; i < 256; i += kT)
        sm.hist2[i] = 0u;
    __syncthreads();
    const uint32_t prefix1 = d1 << (32 - kBits1);
    const uint32_t mask1 = ~0u << (32 - kBits1);
    const uint32_t top_of_bin = prefix1 | ~mask1;
    constexpr int kShift2 = 32 - kBits1 - 8;  // second digit: key bits 20..13
    // whole float4 groups (lo is a multiple of 128, so the slice keeps the
    // row's 16-byte alignment): a warp covers 128 positions = 4 bitmap words
    const int vec_n = (((uintptr_t)s & 15u) == 0) ? len / 4 : 0;
    for (int base = 0; base < vec_n; base += kT * kBatchV) {
        float4 v[kBatchV];
#pragma unroll
        for (int j = 0; j < kBatchV; ++j) {
            const int i4 = base + j * kT + tid;
            v[j] = i4 < vec_n ? __ldcg(reinterpret_cast<const float4 *>(s) + i4)
                              : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        }
#pragma unroll
        for (int j = 0; j < kBatchV; ++j) {
            const int i4 = base + j * kT + tid;
            const int pos0 = 4 * i4;  // within the slice
            const bool live = i4 < vec_n;
            const float f[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
            uint32_t key[4];
            unsigned hitm = 0u, abovem = 0u;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                key[e] = order_key(f[e]);
                const uint32_t dg = key[e] >> (32 - kBits1);
                hitm |= (live && dg == d1) ? (1u << e) : 0u;
                abovem |= (live && dg > d1) ? (1u << e) : 0u;
            }
            unsigned word = abovem << (4 * (lane & 7));
            word |= __shfl_xor_sync(kFull, word, 1);
            word |= __shfl_xor_sync(kFull, word, 2);
            word |= __shfl_xor_sync(kFull, word, 4);
            if ((lane & 7) == 0 && live)
                sm.bitmap[pos0 >> 5] = word;
            if (hitm) {  // at most bin_count <= kCand hits in the row
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    if (hitm & (1u << e)) {
                        const unsigned slot = atomicAdd(&sm.cand_count, 1u);
                        cand_key[slot] = key[e];
                        cand_pos[slot] = lo + pos0 + e;
                        atomicAdd(&sm.hist2[(key[e] >> kShift2) & 0xffu], 1u);
                    }
            }
        }
    }
    __syncthreads();  // whole-word stores above land before the tail ORs into a word
    for (int i = 4 * vec_n + tid; i < len; i += kT) {  // the slice's last few scores
        const uint32_t key = order_key(__ldcg(&s[i]));
        if (key > top_of_bin)
            atomicOr(&sm.bitmap[i >> 5], 1u << (i & 31));
        else if ((key & mask1) == prefix1) {
            const unsigned slot = atomicAdd(&sm.cand_count, 1u);
            cand_key[slot] = key;
            cand_pos[slot] = lo + i;
            atomicAdd(&sm.hist2[(key >> kShift2) & 0xffu], 1u);
        }
    }
    __syncthreads();
    const unsigned own = sm.cand_count;
    cluster.sync();  // every rank's pairs are complete

    if (rank == 0) {
        // gather the other ranks' pairs behind this rank's own, and add their
        // second-digit counts to this rank's, then select
        for (int i = tid; i < 256; i += kT) {
            unsigned t = sm.hist2[i];
            for (int rr = 1; rr < CS; ++rr)
                t += *cluster.map_shared_rank(&sm.hist2[i], rr);
            sm.hist2[i] = t;
        }
        unsigned total = own;
        for (int rr = 1; rr < CS; ++rr) {
            const unsigned cnt = *cluster.map_shared_rank(&sm.cand_count, rr);
            const uint32_t *rk = cluster.map_shared_rank(cand_key, rr);
            const int32_t *rp = cluster.map_shared_rank(cand_pos, rr);
            for (unsigned i = tid; i < cnt; i += kT) {
                cand_key[total + i] = rk[i];
                cand_pos[total + i] = rp[i];
            }
            total += cnt;
        }
        __syncthreads();
        const unsigned warp_max =
            a.warp_select_max > 0 ? (unsigned)a.warp_select_max : kWarpSelectMax;
        bin_cut<NT>(sm, cand_key, cand_pos, total, prefix1, mask1, r1, warp_max);
    }
    cluster.sync();  // the cut is in rank 0's shared memory; rank 0 is done reading the pairs
    const uint32_t T = *cluster.map_shared_rank(&sm.cut[0], 0);
    const int P = (int)*cluster.map_shared_rank(&sm.cut[1], 0);
    for (unsigned i = tid; i < own; i += kT) {  // this rank's own pairs (the first `own`)
        const uint32_t key = cand_key[i];
        const int pos = cand_pos[i];
        if (key > T || (key == T && pos <= P))
            atomicOr(&sm.bitmap[(pos - lo) >> 5], 1u << ((pos - lo) & 31));
    }
    __syncthreads();
    // positions kept by this slice, then their order within the slice
    constexpr int kWordsPerThread = C::kWordsPerThread;
    const int words = (len + 31) / 32;
    const int wpt = (words + kT - 1) / kT;  // the slice's words spread evenly, <= kWordsPerThread
    const int w0 = tid * wpt;
    unsigned w[kWordsPerThread];
    unsigned count = 0;
#pragma unroll
    for (int j = 0; j < kWordsPerThread; ++j) {
        const int wi = w0 + j;
        w[j] = (j < wpt && wi < words) ? sm.bitmap[wi] : 0u;
        count += __popc(w[j]);
    }
    unsigned slice_total;
    unsigned slot = block_exclusive_sum(sm, count, &slice_total);
    if (tid == 0)
        sm.slice_total = slice_total;
    cluster.sync();  // every slice's total is known
    unsigned before = 0;
    for (int rr = 0; rr < rank; ++rr)
        before += *cluster.map_shared_rank(&sm.slice_total, rr);
    cluster.sync();  // no rank leaves while another may still read its shared memory
    const int kcap = a.top_k;
    int32_t *out = a.idx + bg * (size_t)kcap;
    slot += before;
#pragma unroll
    for (int j = 0; j < kWordsPerThread; ++j) {
        unsigned word = w[j];
        while (word) {
            const int bit = __ffs(word) - 1;
            word &= word - 1u;
            if (slot < (unsigned)k)  // exactly k bits are set over all slices
                out[slot] = lo + (w0 + j) * 32 + bit;
            ++slot;
        }
    }
    if (rank == 0) {
        for (int j = k + tid; j < kcap; j += kT)
            out[j] = -1;  // a per-row budget below the row length
        if (a.counts && tid == 0)
            a.counts[bg] = k;
    }
}

// ---------------------------------------------------------------------------
// Coverage budget ("Dynamic Token Coverage", Token Sparse Attention §2: sort
// the tokens by importance and prune the least important ones while their
// cumulative attention mass stays within tau).  Per (batch row, KV head): the
// smallest k such that the k highest-scoring positions hold at least 1 - tau
// of softmax(s) over the row's N_b scores (ties: lower positions first), then
// min(k, kcap).  Mass is reduced by radix descent over the order-preserving
// keys: at each digit level a histogram of counts and of exp(s - max) sums
// finds the digit where the mass accumulated from the top reaches the
// target; at the full key T the last few keys equal to T are counted
// arithmetically.  Every pass streams the row (L2-resident after the
// selection layer wrote it).
constexpr int kCovThreads = 1024;
constexpr int kCovWarps = kCovThreads / 32;

constexpr int kCovCand = 3072;  // (key, mass) pairs of the crossing bin kept in shared memory
constexpr int kCovBatch = 8;    // scores loaded per thread before they are used

struct CovSmem {
    unsigned cnt[kBins1];
    float mass[kBins1];
    float red[kCovWarps];
    float fres[2];      // mass above the chosen digit, mass of the chosen digit
    unsigned ures[3];   // digit, count above it, count of it
    unsigned ccount;
    uint32_t ckey[kCovCand];
    float cmass[kCovCand];
};

// Inverse of order_key.
__device__ __forceinline__ float key_to_float(uint32_t key)
{
    return __uint_as_float((key & 0x80000000u) ? (key & 0x7fffffffu) : ~key);
}

__device__ float cov_block_max(CovSmem &sm, float v)
{
    for (int off = 16; off >= 1; off >>= 1)
        v = fmaxf(v, __shfl_xor_sync(kFull, v, off));
    if ((threadIdx.x & 31) == 0)
        sm.red[threadIdx.x >> 5] = v;
    __syncthreads();
    if (threadIdx.x < 32) {
        float w = sm.red[threadIdx.x];
        for (int off = 16; off >= 1; off >>= 1)
            w = fmaxf(w, __shfl_xor_sync(kFull, w, off));
        if (threadIdx.x == 0)
            sm.fres[0] = w;
    }
    __syncthreads();
    const float r = sm.fres[0];
    __syncthreads();
    return r;
}

// One warp: over bins nb-1 .. 0 (from the top), the first non-empty bin at
// which the mass accumulated from the top reaches `target` (clamped to the
// total, so rounding cannot leave it unreached; failing that, the lowest
// non-empty bin).  Writes the digit, the count and mass above it, and its own
// count and mass to ures / fres.
__device__ void cov_find_digit(CovSmem &sm, int nb, float target)
{
    const int lane = threadIdx.x & 31;
    const int per = nb / 32;  // bins per lane; lane 0 owns the top ones
    float ms = 0.0f;
    unsigned cs = 0;
    for (int i = 0; i < per; ++i) {
        const int bin = nb - 1 - lane * per - i;
        ms += sm.mass[bin];
        cs += sm.cnt[bin];
    }
    float mi = ms;
    unsigned ci = cs;
    for (int off = 1; off < 32; off <<= 1) {
        const float mt = __shfl_up_sync(kFull, mi, off);
        const unsigned ct = __shfl_up_sync(kFull, ci, off);
        if (lane >= off) {
            mi += mt;
            ci += ct;
        }
    }
    const float t = fminf(target, __shfl_sync(kFull, mi, 31));
    const unsigned reach = __ballot_sync(kFull, cs > 0 && mi >= t);
    const int src = reach ? __ffs(reach) - 1 : 31 - __clz(__ballot_sync(kFull, cs > 0));
    if (lane == src) {
        float run = mi - ms, prun = run;
        unsigned crun = ci - cs, pcrun = crun;
        int pick = nb - 1 - lane * per;
        for (int i = 0; i < per; ++i) {
            const int bin = nb - 1 - lane * per - i;
            if (sm.cnt[bin] == 0)
                continue;
            pick = bin;
            prun = run;
            pcrun = crun;
            if (run + sm.mass[bin] >= t)
                break;
            run += sm.mass[bin];
            crun += sm.cnt[bin];
        }
        sm.ures[0] = (unsigned)pick;
        sm.ures[1] = pcrun;
        sm.ures[2] = sm.cnt[pick];
        sm.fres[0] = prun;
        sm.fres[1] = sm.mass[pick];
    }
}

// Reference for exp(s - M): any M >= max(s) keeps every term <= 1 and the
// mass ratios exact.  The selection layer's first-digit histogram gives one
// for free: the largest score of its highest non-empty bin.  NaN when that
// bin is too wide (huge scores) or not finite: then the exact maximum is
// needed.  Every thread of the block must call it (it uses `red`).
template <int NT>
__device__ float cov_reference(const unsigned *gh, float *red)
{
    constexpr int nw = NT / 32;
    int top_bin = -1;
    for (int i = threadIdx.x; i < kBins1; i += NT)
        if (__ldcg(gh + i))
            top_bin = i;
    top_bin = __reduce_max_sync(kFull, top_bin);
    if ((threadIdx.x & 31) == 0)
        red[threadIdx.x >> 5] = __int_as_float(top_bin);
    __syncthreads();
    int tb = -1;
    for (int w = 0; w < nw; ++w)
        tb = max(tb, __float_as_int(red[w]));
    __syncthreads();
    const uint32_t kmin = (uint32_t)(tb < 0 ? 0 : tb) << (32 - kBits1);
    const float M = key_to_float(kmin | (~0u >> kBits1));
    return (isfinite(M) && M - key_to_float(kmin) <= 60.0f) ? M : NAN;
}

// First digit of the coverage descent, spread over several CTAs per row:
// counts and exp(s - M) sums of the top 11 bits of this CTA's part of the
// row, added into the row's global histogram.  Rows whose reference is not
// usable are left to the single-CTA path.
constexpr int kCovPartThreads = 256;
constexpr int kCovPart = kCovPartThreads * 16;  // scores per CTA

__global__ void __launch_bounds__(kCovPartThreads)
coverage_part_kernel(const CoverageArgs a)
{
    __shared__ unsigned cnt[kBins1];
    __shared__ float mass[kBins1];
    __shared__ float red[kCovPartThreads / 32];
    const int part = blockIdx.x, g = blockIdx.y, b = blockIdx.z, tid = threadIdx.x;
    const size_t bg = (size_t)b * a.Hkv + g;
    int n = a.seq_lens[b];
    n = n < 0 ? 0 : (n > a.Nmax ? a.Nmax : n);
    pdl_wait();
    pdl_launch_dependents();
    const int i0 = part * kCovPart;
    if (i0 >= n)
        return;
    const float M = cov_reference<kCovPartThreads>(a.hist + bg * kBins1, red);
    if (isnan(M))
        return;
    for (int i = tid; i < kBins1; i += kCovPartThreads) {
        cnt[i] = 0u;
        mass[i] = 0.0f;
    }
    __syncthreads();
    const float *s = a.scores + bg * (size_t)a.Nmax;
    const int i1 = min(i0 + kCovPart, n);
    float v[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        const int i = i0 + j * kCovPartThreads + tid;
        v[j] = i < i1 ? __ldcg(s + i) : 0.0f;
    }
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        const int i = i0 + j * kCovPartThreads + tid;
        if (i < i1) {
            const unsigned d = order_key(v[j]) >> (32 - kBits1);
            atomicAdd(&cnt[d], 1u);
            atomicAdd(&mass[d], expf(v[j] - M));
        }
    }
    __syncthreads();
    unsigned *gc = a.gcnt + bg * kBins1;
    float *gm = a.gmass + bg * kBins1;
    for (int i = tid; i < kBins1; i += kCovPartThreads)
        if (cnt[i]) {
            atomicAdd(&gc[i], cnt[i]);
            atomicAdd(&gm[i], mass[i]);
        }
}

__global__ void __launch_bounds__(kCovThreads)
coverage_kernel(const CoverageArgs a)
{
    __shared__ CovSmem sm;
    const int g = blockIdx.x, b = blockIdx.y, tid = threadIdx.x;
    const size_t bg = (size_t)b * a.Hkv + g;
    int n = a.seq_lens[b];
    n = n < 0 ? 0 : (n > a.Nmax ? a.Nmax : n);
    const float *s = a.scores + bg * (size_t)a.Nmax;
    pdl_wait();
    pdl_launch_dependents();
    if (n == 0) {
        if (tid == 0)
            a.row_k[bg] = 0;
        return;
    }
    // the reference M the part kernels used (same histogram, same value), or
    // the exact maximum where it is not usable
    float M = a.hist ? cov_reference<kCovThreads>(a.hist + bg * kBins1, sm.red) : NAN;
    const bool have_parts = a.gcnt && !isnan(M);
    if (isnan(M)) {
        float mx = -INFINITY;
        for (int i = tid; i < n; i += kCovThreads)
            mx = fmaxf(mx, __ldcg(s + i));
        M = cov_block_max(sm, mx);
    }

    // Levels after the first run on the crossing bin's elements, gathered into
    // shared memory when they fit, else streamed from the row again.  The
    // loops run in whole warps (f gets a validity flag) so that f can combine
    // lanes with warp collectives.
    bool gathered = false;
    auto for_each = [&](uint32_t mask, uint32_t prefix, auto f) {
        if (gathered) {
            const unsigned cnt = sm.ccount;
            for (unsigned base = 0; base < cnt; base += kCovThreads) {
                const unsigned i = base + tid;
                const bool in = i < cnt && (sm.ckey[i] & mask) == prefix;
                f(in, in ? sm.ckey[i] : 0u, in ? sm.cmass[i] : 0.0f);
            }
        } else {
            // kCovBatch loads in flight per thread before any is used
            for (int base = 0; base < n; base += kCovThreads * kCovBatch) {
                float v[kCovBatch];
#pragma unroll
                for (int j = 0; j < kCovBatch; ++j) {
                    const int i = base + j * kCovThreads + tid;
                    v[j] = i < n ? __ldcg(s + i) : 0.0f;
                }
#pragma unroll
                for (int j = 0; j < kCovBatch; ++j) {
                    const int i = base + j * kCovThreads + tid;
                    const uint32_t key = order_key(v[j]);
                    const bool in = i < n && (key & mask) == prefix;
                    f(in, key, in ? expf(v[j] - M) : 0.0f);
                }
            }
        }
    };
    // Histogram update with the lanes of a warp that hit the same bin
    // combined first: scores crowd into few bins, and one shared-memory atomic
    // per bin and warp instead of one per score removes most of the contention.
    const int lane = tid & 31;
    auto hist_add = [&](bool in, unsigned d, float e) {
        const unsigned grp = __match_any_sync(kFull, in ? d : 0xffffffffu);
        float sum = 0.0f;
#pragma unroll
        for (int src = 0; src < 32; ++src) {
            const float ev = __shfl_sync(kFull, e, src);
            if ((grp >> src) & 1u)
                sum += ev;
        }
        if (in && __ffs(grp) - 1 == lane) {
            atomicAdd(&sm.cnt[d], (unsigned)__popc(grp));
            atomicAdd(&sm.mass[d], sum);
        }
    };

    uint32_t prefix = 0u, mask = 0u;
    unsigned count_above = 0;
    float mass_above = 0.0f, target = 0.0f;
    // digit widths from the top: 11, 8, 8, 5 bits
    for (int level = 0, top = 31; level < 4; ++level) {
        const int width = level == 0 ? kBits1 : (level == 3 ? 5 : 8);
        const int shift = top + 1 - width;
        const unsigned nb = 1u << width;
        if (level == 0 && have_parts) {
            // the part kernels' first-digit histogram; cleared for the next use
            unsigned *gc = a.gcnt + bg * kBins1;
            float *gm = a.gmass + bg * kBins1;
            for (int i = tid; i < (int)nb; i += kCovThreads) {
                sm.cnt[i] = __ldcg(gc + i);
                sm.mass[i] = __ldcg(gm + i);
                gc[i] = 0u;
                gm[i] = 0.0f;
            }
        } else {
            for (int i = tid; i < (int)nb; i += kCovThreads) {
                sm.cnt[i] = 0u;
                sm.mass[i] = 0.0f;
            }
            __syncthreads();
            for_each(mask, prefix, [&](bool in, uint32_t key, float e) {
                hist_add(in, (key >> shift) & (nb - 1u), e);
            });
        }
        __syncthreads();
        if (level == 0) {
            // the whole row's mass: the softmax denominator (relative to M)
            float part = 0.0f;
            for (int i = tid; i < (int)nb; i += kCovThreads)
                part += sm.mass[i];
            for (int off = 16; off >= 1; off >>= 1)
                part += __shfl_xor_sync(kFull, part, off);
            if ((tid & 31) == 0)
                sm.red[tid >> 5] = part;
            __syncthreads();
            if (tid == 0) {
                float L = 0.0f;
                for (int w = 0; w < kCovWarps; ++w)
                    L += sm.red[w];
                sm.fres[0] = L;
            }
            __syncthreads();
            target = (1.0f - a.tau) * sm.fres[0];
            __syncthreads();
        }
        if (tid < 32)
            cov_find_digit(sm, (int)nb, target - mass_above);
        __syncthreads();
        const unsigned d = sm.ures[0];
        count_above += sm.ures[1];
        mass_above += sm.fres[0];
        const unsigned cnt_d = sm.ures[2];
        const float mass_d = sm.fres[1];
        prefix |= d << shift;
        mask |= (nb - 1u) << shift;
        top -= width;
        __syncthreads();
        if (count_above >= (unsigned)a.kcap) {
            // more keys above the cut than the row can hold: the budget is the cap
            if (tid == 0)
                a.row_k[bg] = a.kcap;
            return;
        }
        if (level == 3 || cnt_d == 1u) {
            // every key left equals the chosen one (or there is one): each carries
            // mass_d / cnt_d; take as many as the remaining target needs
            const float each = mass_d / (float)cnt_d;
            const float need = target - mass_above;
            unsigned j = cnt_d;
            if (each > 0.0f && need <= each * (float)cnt_d) {
                const float q = ceilf(need / each);
                j = q < 1.0f ? 1u : (q > (float)cnt_d ? cnt_d : (unsigned)q);
            }
            if (tid == 0) {
                const unsigned kc = count_above + j;
                a.row_k[bg] = (int)(kc < (unsigned)a.kcap ? kc : (unsigned)a.kcap);
            }
            return;
        }
        if (level == 0 && cnt_d <= (unsigned)kCovCand) {
            // one more read of the row: the crossing bin's (key, mass) pairs
            if (tid == 0)
                sm.ccount = 0u;
            __syncthreads();
            for (int base = 0; base < n; base += kCovThreads * kCovBatch) {
                float v[kCovBatch];
#pragma unroll
                for (int j = 0; j < kCovBatch; ++j) {
                    const int i = base + j * kCovThreads + tid;
                    v[j] = i < n ? __ldcg(s + i) : 0.0f;
                }
#pragma unroll
                for (int j = 0; j < kCovBatch; ++j) {
                    const int i = base + j * kCovThreads + tid;
                    const uint32_t key = order_key(v[j]);
                    if (i < n && (key & mask) == prefix) {
                        const unsigned slot = atomicAdd(&sm.ccount, 1u);
                        if (slot < (unsigned)kCovCand) {  // exactly cnt_d land; the bound guards memory
                            sm.ckey[slot] = key;
                            sm.cmass[slot] = expf(v[j] - M);
                        }
                    }
                }
            }
            __syncthreads();
            if (sm.ccount > (unsigned)kCovCand)
                sm.ccount = kCovCand;  // unreachable: the histogram counted cnt_d of them
            __syncthreads();
            gathered = true;
        }
    }
}

template <int NT>
constexpr size_t topk_smem_bytes()
{
    return sizeof(TopkSmem<NT>) + (size_t)TopkCfg<NT>::kCand * (sizeof(uint32_t) + sizeof(int32_t));
}

static_assert(kSubHists * kBins1 <= 2 * TopkCfg<512>::kCand, "pass-1 sub-histograms fit in the candidate area");
static_assert(2 * (topk_smem_bytes<512>() + 1024) <= 228 * 1024, "two 512-thread CTAs fit one SM");

template <int NT>
cudaError_t launch_topk_nt(const TopkArgs &a, int batch, bool pdl, cudaStream_t stream)
{
    constexpr size_t smem = topk_smem_bytes<NT>();
    static bool configured[64] = {false};  // the smem opt-in is per device
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= 64 || !configured[dev]) {
        e = cudaFuncSetAttribute(topk_kernel<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem);
        if (e != cudaSuccess)
            return e;
        if (dev >= 0 && dev < 64)
            configured[dev] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)a.Hkv, (unsigned)batch);
    cfg.blockDim = dim3(NT);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, topk_kernel<NT>, a);
}

template <int CS>
cudaError_t launch_topk_cluster(const TopkArgs &a, int batch, bool pdl, cudaStream_t stream)
{
    constexpr size_t smem = topk_smem_bytes<kClusterNT>();
    static bool configured[64] = {false};  // the smem opt-in is per device
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= 64 || !configured[dev]) {
        e = cudaFuncSetAttribute(topk_cluster_kernel<CS>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess)
            return e;
        if (dev >= 0 && dev < 64)
            configured[dev] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)CS, (unsigned)a.Hkv, (unsigned)batch);  // cluster dims: compiled in
    cfg.blockDim = dim3(kClusterNT);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, topk_cluster_kernel<CS>, a);
}

}  // namespace

cudaError_t launch_topk(const TopkArgs &a, int batch, int threads, int cluster, bool pdl,
                        cudaStream_t stream)
{
    if (cluster == 2 || cluster == 4 || cluster == 8) {
        return cluster == 8   ? launch_topk_cluster<8>(a, batch, pdl, stream)
               : cluster == 4 ? launch_topk_cluster<4>(a, batch, pdl, stream)
                              : launch_topk_cluster<2>(a, batch, pdl, stream);
    }
    // Default 1024: with more rows than SMs, two 512-thread CTAs per SM take
    // every register of the SM, and the next layer's attention CTAs, launched
    // early by programmatic dependent launch, then find no room next to them;
    // in a CUDA-graph step that cost ~150 us per selection layer (measured at
    // batch 32 x 8 KV heads) against ~3 us gained by the top-k itself.
    if (threads != 512)
        threads = 1024;
    return threads == 512 ? launch_topk_nt<512>(a, batch, pdl, stream)
                          : launch_topk_nt<1024>(a, batch, pdl, stream);
}

cudaError_t launch_coverage(const CoverageArgs &a, int batch, bool pdl, cudaStream_t stream)
{
    if (a.gcnt && a.hist) {
        cudaLaunchConfig_t pc = {};
        pc.gridDim = dim3((unsigned)((a.Nmax + kCovPart - 1) / kCovPart), (unsigned)a.Hkv,
                          (unsigned)batch);
        pc.blockDim = dim3(kCovPartThreads);
        pc.stream = stream;
        cudaLaunchAttribute pattr[1];
        pattr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        pattr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
        pc.attrs = pattr;
        pc.numAttrs = 1;
        cudaError_t e = cudaLaunchKernelEx(&pc, coverage_part_kernel, a);
        if (e != cudaSuccess)
            return e;
        pdl = true;  // the row kernel follows the part kernel
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)a.Hkv, (unsigned)batch);
    cfg.blockDim = dim3(kCovThreads);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, coverage_kernel, a);
}

}  // namespace td
