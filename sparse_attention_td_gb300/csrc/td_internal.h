// td_internal.h -- kernel arguments and launchers shared by the library's
// translation units (not part of the public C ABI).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace td {

constexpr int kHeadDim = 128;          // only head_dim supported
constexpr int kAttnThreads = 256;      // 8 warps
constexpr int kAttnWarps = kAttnThreads / 32;
constexpr int kTokPerHalf = 4;         // tokens a half-warp handles per round
constexpr int kTokPerRound = kAttnWarps * 2 * kTokPerHalf;  // 64 tokens per CTA round
constexpr int kChunkGranule = 16;      // split lengths are multiples of this many tokens
constexpr int kMaxSplits = 256;        // splits per (batch, KV head)
constexpr int kMaxClusterSplits = 16;  // splits a cluster merge can take (non-portable above 8)
constexpr int kPortableClusterSplits = 8;  // the split counts merged through a cluster by default
constexpr int kMaxSplitCtas = 8192;    // cap on batch * kv_heads * splits for partials
constexpr int kMaxSparseChunk = 2048;  // index entries one sparse CTA stages in shared memory
constexpr int kMaxTopK = kMaxSplits * kMaxSparseChunk;
constexpr int kTopkCandidates = 16384;  // (key, position) pairs a 1024-thread top-k CTA holds in shared memory
constexpr int kSelectBits = 11;         // first radix digit of the top-k select (key bits 31..21)
constexpr int kSelectBins = 1 << kSelectBits;
constexpr int kTopkBitmapBits = 1 << 18; // rows up to this length are compacted through a bitmap

constexpr uint32_t kFlagIndexOutOfRange = 0x1u;
constexpr uint32_t kFlagSeqLenOutOfRange = 0x2u;
constexpr uint32_t kFlagWaitTimeout = 0x4u;  // a bounded wait for an async copy gave up

// A TMA tensor map (the driver's CUtensorMap: 128 opaque bytes, 64-byte aligned).
struct alignas(64) TmaDesc {
    unsigned char bytes[128];
};

// One attention launch (full or sparse).  Partials are struct-of-arrays over
// (batch*kv_head, split, head-in-group[, dim]) with split stride `nsplit`.
struct AttnArgs {
    const uint16_t *q;       // [B][Hq][128] bf16 bits
    const uint16_t *k;       // [B][Hkv][Nmax][128]
    const uint16_t *v;
    const int32_t *seq_lens; // [B]
    const int32_t *idx;      // sparse: [B][Hkv][top_k]
    uint16_t *out;           // [B][Hq][128]
    float *out_f32;          // optional
    float *scores;           // select: [B][Hkv][Nmax]
    unsigned *hist;          // select: [B*Hkv][kSelectBins] first-digit histogram (zero on entry)
    float *part_m;           // [B*Hkv][nsplit][G]  running max (log2 units)
    float *part_l;           // [B*Hkv][nsplit][G]  softmax denominator
    float *part_o;           // [B*Hkv][nsplit][G][128] un-normalised output
    uint32_t *tickets;       // [B*Hkv] arrival counters, zero between launches
    uint32_t *status;        // device status word
    int Hq, Hkv, Nmax, top_k;
    int idx_dep;             // sparse: the index set may be written by the previous kernel
    int chunk;               // tokens (full) or index entries (sparse) per split
    int nsplit;              // gridDim.x
    int prefetch;            // full layers: rounds ahead whose rows each warp prefetches into L2 (0: none)
    int early_trigger;       // >0: a CTA lets the next kernel launch at the start of its round
                             // n_rounds - early_trigger (ring, register-streamed, cp.async-staged
                             // sparse and 16-token full kernels; after its wait for the previous
                             // kernel); 0: after the loop
    int interleave;          // full layers (tensor cores with 16 tokens per warp, CUDA cores
                             // register-streamed): the splits of a (batch row, KV head) take its
                             // 64-token rounds in turn instead of one chunk each
    int wait_limit_us;       // staged full layers: microseconds before a stage wait gives up (0: 1 s)
    int wait_test;           // staged full layers: each CTA's first wait polls a barrier nothing
                             // arrives on (tests of the failure report); 0 in normal use
    float scale;             // softmax scale (natural-log units)
    int sk_ctas;             // sparse, stream-K partition (tensor cores, 16 tokens per warp): the
                             // CTAs (1D grid) sharing the layer's rounds evenly; 0: not used
    int sk_units;            // with sk_ctas: (batch row, KV head) pairs, B * Hkv
    int tma_rows;            // sparse, row gathers: rows of the maps (B * Hkv * Nmax)
    TmaDesc tma_k, tma_v;    // sparse, row gathers: maps over the K / V cache rows
};

struct TopkArgs {
    const float *scores;     // [B][Hkv][Nmax]
    unsigned *hist;          // [B*Hkv][kSelectBins] from the attention kernel, or null; zeroed after use
    const int32_t *seq_lens; // [B]
    int32_t *idx;            // [B][Hkv][top_k]
    uint32_t *status;
    const int32_t *row_k;    // [B*Hkv] per-row budget (<= top_k), or null: top_k for every row
    int32_t *counts;         // [B*Hkv] positions selected per row (min(k, N_b)), or null
    int Hkv, Nmax, top_k;
    int warp_select_max;     // threshold bins up to this many pairs finish in one warp (0: the default, 256)
};

// Coverage budget per (batch row, KV head): row_k[bg] = min(kcap, smallest k
// whose top-k scores hold >= 1 - tau of softmax(scores) over the row).
struct CoverageArgs {
    const float *scores;     // [B][Hkv][Nmax]
    const unsigned *hist;    // [B*Hkv][kSelectBins] first-digit counts of the scores, or null
    const int32_t *seq_lens; // [B]
    int32_t *row_k;          // [B*Hkv] out
    unsigned *gcnt;          // [B*Hkv][kSelectBins] first-digit counts (zero on entry), or null
    float *gmass;            // [B*Hkv][kSelectBins] first-digit mass sums (zero on entry)
    int Hkv, Nmax, kcap;
    float tau;
};

// G = query heads per KV head (1, 2, 4, 8).
// cluster: merge the splits through a thread-block cluster (requires
// a.nsplit <= kMaxClusterSplits); otherwise through global partials.
// staged: K/V rows reach shared memory through a ring of stages (ignored when
// cluster is set): 1 by bulk copies (full) or per-thread cp.async (sparse),
// 2 (sparse) by TMA row gathers through a.tma_k / a.tma_v; 0 register-streamed.
// pdl: the launch may overlap the tail of the kernel before it on the stream
// (programmatic dependent launch); only for a kernel whose predecessor is a
// kernel of the same call.
cudaError_t launch_attention(int G, bool sparse, bool select, bool cluster, int staged,
                             const AttnArgs &a, int batch, bool pdl, cudaStream_t stream);
// threads: 1024 or 512 threads per row's CTA (0: 1024).  cluster: 2, 4 or 8
// CTAs of 1024 threads per row, merged through distributed shared memory;
// other values: one CTA per row.
cudaError_t launch_topk(const TopkArgs &a, int batch, int threads, int cluster, bool pdl,
                        cudaStream_t stream);
cudaError_t launch_coverage(const CoverageArgs &a, int batch, bool pdl, cudaStream_t stream);

// KV append of up to kAppendLayers layers in one launch: for each layer l,
// rows k_new[l] / v_new[l] [B][Hkv][128] written at position seq_lens[b]-1 of
// k[l] / v[l].
constexpr int kAppendLayers = 32;
struct AppendBatch {
    uint16_t *k[kAppendLayers];
    uint16_t *v[kAppendLayers];
    const uint16_t *k_new[kAppendLayers];
    const uint16_t *v_new[kAppendLayers];
};
cudaError_t launch_kv_append(const AppendBatch &layers, int num_layers, const int32_t *seq_lens,
                             int batch, int Hkv, int Nmax, cudaStream_t stream);

// counts[b*Hkv + g] = |a[b][g] ∩ b[b][g]| over two ascending, -1-padded index rows.
cudaError_t launch_index_overlap(const int32_t *a, const int32_t *b, int rows, int top_k,
                                 int32_t *counts, cudaStream_t stream);

// Read probe (measurement aid): the K/V row reads of one attention launch
// with the given split plan, folded into an XOR; idx == null reads the
// contiguous rows of a full layer.
struct ProbeArgs {
    const uint16_t *k, *v;
    const int32_t *seq_lens;
    const int32_t *idx;      // sparse: [B][Hkv][top_k], or null for a full layer
    uint32_t *sink;          // sink_words words
    int sink_words;
    int Hkv, Nmax, top_k, chunk, nsplit;
};
cudaError_t launch_probe_reads(const ProbeArgs &a, int batch, cudaStream_t stream);

// Tensor-core attention (mma.sync over a KV head's G query heads) for
// G = 4 and 8: same arguments and results as launch_attention (no cluster
// merge, register-fed fragments).  tokens: tokens a warp takes per round,
// 8 (CTAs of 8 warps) or 16 (CTAs of 4 warps); 32: 16 per round with two
// rounds in flight per warp.
bool mma_supported(int G);
cudaError_t launch_attention_mma(int G, bool sparse, bool select, int tokens, const AttnArgs &a,
                                 int batch, bool pdl, cudaStream_t stream);
int attention_mma_ctas_per_sm(int G, bool sparse, bool select, int tokens);

// Preferred shared-memory carveout (percent, -1 = driver default) for later attention launches.
void set_attention_carveout(int percent);

// Resident CTAs per SM of one attention instantiation (occupancy query).
int attention_ctas_per_sm(int G, bool sparse, bool select, int staged);

}  // namespace td
