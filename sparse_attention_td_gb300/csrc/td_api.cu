// td_api.cu -- the C ABI of include/td.h: argument validation, workspace
// layout, split planning, the per-step layer scheduler and CUDA-graph plans.
//
// The layer scheduler follows the decode step of the TidalDecode paper
// review (§三 Figure 2): full layers run the attention kernel, selection
// layers run it with score emission followed by the top-k kernel (which
// overwrites the resident index buffer), and PPSA layers run the sparse
// attention kernel over the most recent selection (§三 "Position Persistent
// Sparse Attention": later layers reuse the selected positions).
#include <cuda.h>  // tensor-map types only: the encoder is reached through the runtime
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <mutex>
#include <new>
#include <vector>

#include "../../include/td.h"
#include "td_internal.h"

namespace {

using td::kHeadDim;

struct Tuning {
    int full_ctas_per_sm = 0;    // 0 = occupancy query
    int sparse_ctas_per_sm = 0;
    int full_waves = 0;          // 0 = auto (see plan_splits)
    int sparse_waves = 1;
    int sparse_splits = 0;       // splits per (batch row, KV head) of sparse launches (0: from the
                                 // CTAs per SM and waves above)
    int max_splits = td::kMaxSplits;
    int cluster = 0;             // 1: merge up to kPortableClusterSplits splits through a cluster
    int topk_threads = 0;        // 1024 or 512 threads per row; 0: automatic (topk_threads_for)
    int full_staged = -1;        // 1: full / full+select kernels stage K/V through shared memory
                                 // (bulk copies); 0: register-streamed; -1: staged when G >= 4
    int sparse_staged = -1;      // CUDA-core sparse kernels: 1 stage the gathered rows through
                                 // shared memory (per-thread cp.async ring); 2 through TMA row
                                 // gathers (tile::gather4); 0 register-streamed; -1 auto (1 for
                                 // small layers, see staged_for)
    int mma = -1;                // 1 / -1 (default): tensor-core kernels for G = 4, 8; 0: CUDA cores
    int full_prefetch = -1;      // full / full+select layers: rounds ahead each warp prefetches into
                                 // L2 (register-streamed kernels); -1: 1 on the tensor cores, else 0
    int topk_warp_max = 0;       // top-k threshold bins up to this size finish in one warp (0: 256)
    int topk_cluster = 0;        // CTAs per top-k row of a selection layer: 0 auto, 1, 2, 4, 8
    int pdl = 1;                 // 0: no programmatic dependent launch between a call's kernels
    int topk_pdl = 1;            // 0: the top-k kernel waits for its attention kernel in stream order
    int sparse_stream_k = 0;     // tensor-core sparse layers: 1 splits the layer's rounds evenly over
                                 // whole waves of CTAs (stream-K), 0 one CTA per split
    int mma_full_tokens = 16;    // tensor-core full / full+select kernels: tokens per warp per round
    int mma_sparse_tokens = 0;   // tensor-core sparse kernels: tokens per warp per round (8, 16, or
                                 // 32 = 16 with two rounds in flight, 64 = rounds staged in shared
                                 // memory); 0: 64
    int full_interleave = 1;     // full layers (tensor cores with 16 tokens per warp, or CUDA cores
                                 // register-streamed): 1 the splits of a (batch row, KV head)
                                 // take its 64-token rounds in turn, 0 one contiguous chunk each
    // Rounds before the end of its last round at which a CTA of the ring,
    // register-streamed, cp.async-staged sparse or 16-token full kernel lets
    // the next kernel launch
    // (always after its own wait for the previous kernel, so at most one more
    // grid is launched ahead); 0: after the last round.  Measured on GB300
    // (graph steps), 0 / 1 / 2 / 3 / 4 / 6: serving k=1024 1804 / 1793 /
    // 1784 / 1770 / 1767 / 1781 us, 32K 755 / 747 / 747 / 745 / 744 / 745 us,
    // 100K 1419 / 1414 / 1415 / 1414 / 1412 / 1414 us, serving k=4096
    // 3844 / 3841 / 3826 / 3813 / - / 3808 us, 10K 282.5 -> 280.4 us (4, with
    // the cp.async-staged sparse layers).
    int early_trigger = 4;
    int host_copy = 1;           // host-buffer plans: 1 copy kernels in the launch chain (see
                                 // StepIo), 0 copy-engine copies only
    int wait_limit_us = 0;       // staged full layers: microseconds a stage wait may take before it
                                 // gives up and the launch reports TD_FLAG_WAIT_TIMEOUT (0: 1 s)
    int wait_test = 0;           // 1: each staged full-layer CTA's first wait polls a barrier that
                                 // nothing arrives on, so it runs out (failure-report tests)
};
Tuning g_tuning;
const Tuning kDefaultTuning;

// Measured on GB300: staging pays for the grouped-query full kernels (G >= 4,
// issue-bound at two CTAs per SM) and for none of the others.
// Measured on GB300: the tensor-core kernels take 6-9% off grouped-query
// full layers and match the CUDA-core ones on sparse layers.
bool mma_for(int G) { return g_tuning.mma != 0 && td::mma_supported(G); }

// Measured on GB300: the 16-token tensor-core kernel (CTAs of 4 warps, both
// MMA row groups) takes 2-6% off full and full+select layers; on sparse
// layers it is 9-30% slower than the 8-token kernel, which stays there.
// Measured on GB300: prefetching the next round's K/V lines into L2 takes
// 10% off the tensor-core full layers (32K, G = 4) and costs 5% on the MHA
// full layers at 10K.
int prefetch_for(int G)
{
    return g_tuning.full_prefetch < 0 ? (mma_for(G) ? 1 : 0) : g_tuning.full_prefetch;
}

// Measured on GB300 (graph steps): sparse layers staged through the
// shared-memory ring (its first round requested before the wait for the
// previous kernel) beat the 8-token register kernel on every grouped-query
// workload once the ring has two stages: serving batch k = 256 (one 256-row
// CTA per pair) 1279.8 -> 1237.5 us.  With three stages the ring won only
// where a pair's rows are split over several CTAs (32K: 765 -> 756 us) or
// CTAs gather >= 1024 rows (serving k = 1024: 1861 -> 1830 us; k = 4096:
// 4094 -> 3954 us) and lost 0.4-3 us a layer at k = 256.

// Tokens per warp per round of a tensor-core launch (64: the sparse ring
// kernel; the split plan is the same for every sparse tiling).
int mma_tokens_for(bool sparse)
{
    if (!sparse)
        return g_tuning.mma_full_tokens;
    if (g_tuning.mma_sparse_tokens > 0)
        return g_tuning.mma_sparse_tokens;
    return 64;
}

int device_sm_count();

// How a CUDA-core launch gets its K/V rows (0 registers, 1 staged, 2 TMA
// row gathers for sparse layers).  Measured on GB300 (graph step), sparse
// layers: staging through a per-thread cp.async ring takes the 10K MHA step
// from 316 to 289 us, where every CTA of the register plan would gather one
// round (64 rows) or less; on longer CTAs (100K: ~3.5 rounds) it costs 2%.
int staged_for(const td_shape &s, bool sparse, long n_total)
{
    const int G = s.num_q_heads / s.num_kv_heads;
    if (!sparse)
        return (g_tuning.full_staged < 0 ? G >= 4 : g_tuning.full_staged > 0) ? 1 : 0;
    if (g_tuning.sparse_staged >= 0)
        return g_tuning.sparse_staged;
    const long units = (long)s.batch * s.num_kv_heads;
    const long slots = (long)device_sm_count() * td::attention_ctas_per_sm(G, true, false, 0);
    return units * n_total <= slots * td::kTokPerRound ? 1 : 0;
}


constexpr size_t kAlign = 256;
inline size_t align_up(size_t x) { return (x + kAlign - 1) & ~(kAlign - 1); }
inline bool aligned(const void *p, size_t a) { return ((uintptr_t)p % a) == 0; }
inline long ceil_div(long a, long b) { return (a + b - 1) / b; }

// cuTensorMapEncodeTiled, reached through the runtime (the library does not
// link the driver library itself); null if the driver does not provide it.
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_tiled()
{
    static EncodeTiledFn fn = [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            p = nullptr;
        return (EncodeTiledFn)p;
    }();
    return fn;
}

// Tensor map over a cache's rows for TMA row gathers: a 2D bf16 tensor of
// `rows` rows of 128 values (256-byte stride), box 128 x 1 (one row: the
// only box height a tile::gather4 copy takes), no swizzle (a half-warp reads
// a whole 256-byte row, so the stage layout has no bank conflicts), zero fill
// for rows past the end.
bool encode_row_map(td::TmaDesc *out, const void *base, long rows)
{
    static_assert(sizeof(td::TmaDesc) == sizeof(CUtensorMap), "opaque tensor-map size");
    EncodeTiledFn fn = encode_tiled();
    if (!fn || rows < 1 || rows >= (1L << 31) || !aligned(base, 16))
        return false;
    const cuuint64_t dims[2] = {(cuuint64_t)kHeadDim, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)kHeadDim * 2};
    const cuuint32_t box[2] = {(cuuint32_t)kHeadDim, 1};
    const cuuint32_t elem[2] = {1, 1};
    return fn(reinterpret_cast<CUtensorMap *>(out), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
              const_cast<void *>(base), dims, strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Largest split count a launch of `n_total` tokens/entries may use.
int split_cap(long units, long n_total, bool sparse)
{
    long cap = g_tuning.max_splits;
    if (cap > td::kMaxSplits)
        cap = td::kMaxSplits;
    const long by_len = ceil_div(n_total > 0 ? n_total : 1, td::kTokPerRound);
    if (cap > by_len)
        cap = by_len;
    const long by_ctas = td::kMaxSplitCtas / units;
    if (cap > by_ctas)
        cap = by_ctas;
    if (cap < 1)
        cap = 1;
    if (sparse) {  // a sparse CTA stages at most kMaxSparseChunk entries
        const long need = ceil_div(n_total > 0 ? n_total : 1, td::kMaxSparseChunk);
        if (cap < need)
            cap = need;
    }
    return (int)cap;
}

// Partial-result capacity in (batch*kv_head, split) slots: covers every split
// count split_cap can return, for any tuning.
long partial_slots(const td_shape &s, int top_k)
{
    const long units = (long)s.batch * s.num_kv_heads;
    long most = 1;
    // Full launches: at most min(kMaxSplits, ceil(N/64), 8192/units) splits.
    long full = ceil_div(s.max_seq_len > 0 ? s.max_seq_len : 1, td::kTokPerRound);
    if (full > td::kMaxSplits) full = td::kMaxSplits;
    long by_ctas = td::kMaxSplitCtas / units;
    if (by_ctas < 1) by_ctas = 1;
    if (full > by_ctas) full = by_ctas;
    if (full > most) most = full;
    if (top_k > 0) {
        long sp = ceil_div(top_k, td::kTokPerRound);
        if (sp > td::kMaxSplits) sp = td::kMaxSplits;
        if (sp > by_ctas) sp = by_ctas;
        const long need = ceil_div(top_k, td::kMaxSparseChunk);
        if (sp < need) sp = need;
        if (sp > most) most = sp;
    }
    return units * most;
}

struct WsLayout {
    size_t status, tickets, part_m, part_l, part_o, scores, hist, row_k, cov_cnt, cov_mass, total;
};

WsLayout ws_layout(const td_shape &s, int top_k)
{
    const int G = s.num_q_heads / s.num_kv_heads;
    const size_t units = (size_t)s.batch * s.num_kv_heads;
    const size_t slots = (size_t)partial_slots(s, top_k);
    WsLayout w{};
    size_t off = 0;
    w.status = off;
    off = align_up(off + sizeof(uint32_t));
    w.tickets = off;
    off = align_up(off + units * sizeof(uint32_t));
    w.part_m = off;
    off = align_up(off + slots * G * sizeof(float));
    w.part_l = off;
    off = align_up(off + slots * G * sizeof(float));
    w.part_o = off;
    off = align_up(off + slots * G * kHeadDim * sizeof(float));
    w.scores = off;
    if (top_k > 0)
        off = align_up(off + units * (size_t)s.max_seq_len * sizeof(float));
    w.hist = off;  // first-digit histograms of a selection layer (kept zero between uses)
    if (top_k > 0)
        off = align_up(off + units * (size_t)td::kSelectBins * sizeof(unsigned));
    w.row_k = off;  // per-row budgets of a coverage selection
    if (top_k > 0)
        off = align_up(off + units * sizeof(int32_t));
    w.cov_cnt = off;  // first-digit count / mass histograms of a coverage selection (kept zero)
    if (top_k > 0)
        off = align_up(off + units * (size_t)td::kSelectBins * sizeof(unsigned));
    w.cov_mass = off;
    if (top_k > 0)
        off = align_up(off + units * (size_t)td::kSelectBins * sizeof(float));
    w.total = off;
    return w;
}

td_status check_shape(const td_shape *s)
{
    if (!s)
        return TD_ERR_INVALID_ARG;
    if (s->batch < 1 || s->num_q_heads < 1 || s->num_kv_heads < 1 || s->max_seq_len < 1)
        return TD_ERR_INVALID_ARG;
    if (s->num_q_heads % s->num_kv_heads)
        return TD_ERR_INVALID_ARG;
    if (!isfinite(s->scale) || s->scale < 0.0f)
        return TD_ERR_INVALID_ARG;
    const int G = s->num_q_heads / s->num_kv_heads;
    if (s->head_dim != kHeadDim)
        return TD_ERR_UNSUPPORTED_SHAPE;
    if (G != 1 && G != 2 && G != 4 && G != 8)
        return TD_ERR_UNSUPPORTED_SHAPE;
    if (s->batch > 65535 || s->num_kv_heads > 65535)
        return TD_ERR_UNSUPPORTED_SHAPE;
    return TD_OK;
}

float effective_scale(const td_shape &s)
{
    return s.scale != 0.0f ? s.scale : 1.0f / sqrtf((float)s.head_dim);
}

int device_sm_count();

// CTAs per row of a top-k selection: a cluster of CS CTAs per row when rows
// are long (at least kMinClusterRow positions), few enough for rows x CS CTAs
// to fit one wave, and each CTA still scans at least kMinClusterSlice
// positions; else one CTA per row.  Measured on GB300 (graph step): clusters
// of 4 take 10 us off each 100K selection layer (clusters of 2 instead: step
// 1401.8 -> 1423.1 us); at 10K they cost 4.6 us a step, since the cluster's
// CTAs fill their SMs and the next layer's CTAs cannot start early beside
// them.  At 32K they cost 5-19 us while the sparse layers after them were
// planned with a CTA for every slot; with the whole-round sparse plan, which
// leaves slots free, clusters of 2 take 739.3 -> 730.9 us (4: 731.9 us).
constexpr int kMinClusterRow = 32768;
constexpr int kMinClusterSlice = 16384;
int topk_cluster_for(const td_shape &s)
{
    if (g_tuning.topk_cluster > 0)
        return g_tuning.topk_cluster;
    const long rows = (long)s.batch * s.num_kv_heads;
    if (s.max_seq_len < kMinClusterRow)
        return 1;
    for (int cs = 8; cs >= 2; cs /= 2)
        if (rows * cs <= device_sm_count() && s.max_seq_len / cs >= kMinClusterSlice)
            return cs;
    return 1;
}

int device_sm_count()
{
    static std::mutex mu;
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return 152;
    std::lock_guard<std::mutex> lock(mu);
    if (!cached[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            n = 152;
        cached[dev] = n;
    }
    return cached[dev];
}

// Splits and per-split chunk for one launch.
void plan_splits(const td_shape &s, long n_total, bool sparse, bool select, int &nsplit, int &chunk)
{
    const int G = s.num_q_heads / s.num_kv_heads;
    const long units = (long)s.batch * s.num_kv_heads;
    int per_sm = sparse ? g_tuning.sparse_ctas_per_sm : g_tuning.full_ctas_per_sm;
    int resident = per_sm;  // CTAs of the launched kernel that fit one SM
    if (per_sm <= 0) {
        const int staged = mma_for(G) ? 0 : staged_for(s, sparse, n_total);
        per_sm = mma_for(G) ? td::attention_mma_ctas_per_sm(G, sparse, select, mma_tokens_for(sparse))
                            : td::attention_ctas_per_sm(G, sparse, select, staged);
        resident = per_sm;
        // Measured on GB300 (graph step): register-streamed sparse layers
        // planned one CTA per SM below the 4+ that fit leave a slot for the
        // next layer's CTAs to start early (100K MHA step 1438 -> 1426 us);
        // at 2 per SM the launch loses half its warps and is slower.  (One-wave
        // sparse plans now take the whole-round rule below instead.)
        if (sparse && !mma_for(G) && staged == 0 && per_sm >= 4)
            per_sm -= 1;
    }
    const long slots = (long)device_sm_count() * per_sm;  // resident CTAs per wave
    int waves = sparse ? g_tuning.sparse_waves : g_tuning.full_waves;
    // One wave of long CTAs when the pairs are few; more, shorter CTAs balance
    // ragged lengths otherwise.  Measured on GB300 (serving batch, 256 pairs of
    // 8K-16K tokens): 3 waves best for the CUDA-core kernels; 4 for the
    // tensor-core full kernels (full layer 253.6 -> 241.1 us, step -3%; 2 and
    // 6 waves slower).
    if (waves <= 0)
        waves = units * 2 <= slots ? 1 : (mma_for(G) && !sparse ? 4 : 3);
    const long target = slots * waves;
    const int cap = split_cap(units, n_total, sparse);
    const long len = n_total > 0 ? n_total : 1;
    if (sparse && waves == 1 && g_tuning.sparse_splits <= 0) {
        // One wave of sparse CTAs, each of whole 64-entry rounds: the fewest
        // rounds a CTA can take within one wave at the kernel's occupancy,
        // then the fewest splits that still take no more.  Measured on GB300
        // (graph steps): 100K (MHA, k = 4096) 16 splits of 4 rounds 1398.5 us
        // against 14 of 4.75 (the rule before) 1408.3 us, 19 of 3.4 1423.2 us
        // and 13 of 5 1410.8 us; 32K (k = 2048) 8 splits of 4 rounds 738.5 us
        // against 9 of 3.6 745.0 us; 4 to 6 splits and 10 or more (a second
        // wave) slower at both.
        long most = (long)device_sm_count() * resident / units;
        if (most > cap) most = cap;
        if (most < 1) most = 1;
        long ch = ceil_div(ceil_div(len, most), td::kTokPerRound) * td::kTokPerRound;
        if (ch > td::kMaxSparseChunk)
            ch = td::kMaxSparseChunk;
        nsplit = (int)ceil_div(len, ch);
        chunk = (int)ch;
        return;
    }
    long want = target / units;  // whole waves: never spill a few CTAs into an extra wave
    if (sparse && g_tuning.sparse_splits > 0)
        want = g_tuning.sparse_splits;
    if (want < 1) want = 1;
    if (want > cap) want = cap;
    long ch = ceil_div(ceil_div(len, want), td::kChunkGranule) * td::kChunkGranule;
    if (sparse && ch > td::kMaxSparseChunk)
        ch = td::kMaxSparseChunk;
    long ns = ceil_div(len, ch);
    if (ns > cap) {  // rounding pushed past the cap: widen the chunk instead
        ch = ceil_div(ceil_div(len, cap), td::kChunkGranule) * td::kChunkGranule;
        ns = ceil_div(len, ch);
    }
    nsplit = (int)ns;
    chunk = (int)ch;
}

// Threads per top-k CTA of a selection over this shape (one CTA per row);
// next_mode: the mode of the layer launched right after it in the same call
// (-1: none).  512-thread CTAs, two per SM, take more rows than SMs in one
// wave (a lone launch: 68.2 -> 65.0 us on the serving batch), but they leave
// no registers for the next kernel's CTAs to start early beside them, which
// matters unless that kernel needs more than one wave of CTAs anyway.
// Measured on GB300 (serving batch, two-stage sparse ring, graph steps): 1024
// threads against 512 at k = 256 1237.3 / 1301.6 us and k = 1024 1695.2 /
// 1750.7 us (one wave of sparse CTAs after them); at k = 4096 (two splits a
// pair, 1.7 waves) 3776.8 / 3757.7 us; before full layers (selection at
// every layer) 8681 / 10648 us.
int topk_threads_for(const td_shape &s, int top_k, int next_mode)
{
    if (g_tuning.topk_threads > 0)
        return g_tuning.topk_threads;
    const long rows = (long)s.batch * s.num_kv_heads;
    if (rows <= device_sm_count())
        return 1024;
    if (next_mode < 0)
        return 512;
    if (next_mode != TD_MODE_SPARSE)
        return 1024;
    int nsplit = 0, chunk = 0;
    plan_splits(s, top_k, true, false, nsplit, chunk);
    const int G = s.num_q_heads / s.num_kv_heads;
    int per_sm = g_tuning.sparse_ctas_per_sm;
    if (per_sm <= 0)
        per_sm = mma_for(G) ? td::attention_mma_ctas_per_sm(G, true, false, mma_tokens_for(true))
                            : td::attention_ctas_per_sm(G, true, false, staged_for(s, true, top_k));
    return rows * nsplit > (long)device_sm_count() * per_sm ? 512 : 1024;
}

struct Ctx {
    td_shape shape;
    int G;
    float scale;
    WsLayout ws;
    char *wsb;
};

td_status make_ctx(const td_shape *shape, int top_k, void *ws, size_t ws_bytes, Ctx &c)
{
    td_status st = check_shape(shape);
    if (st)
        return st;
    if (top_k < 0 || top_k > shape->max_seq_len)
        return TD_ERR_INVALID_ARG;
    if (top_k > td::kMaxTopK)
        return TD_ERR_UNSUPPORTED_SHAPE;
    if (!ws || !aligned(ws, kAlign))
        return TD_ERR_INVALID_ARG;
    c.shape = *shape;
    c.G = shape->num_q_heads / shape->num_kv_heads;
    c.scale = effective_scale(*shape);
    c.ws = ws_layout(*shape, top_k);
    if (ws_bytes < c.ws.total)
        return TD_ERR_WORKSPACE_TOO_SMALL;
    c.wsb = (char *)ws;
    return TD_OK;
}

td::AttnArgs base_args(const Ctx &c, const void *q, const void *k, const void *v,
                       const int32_t *seq_lens, void *out, float *out_f32)
{
    td::AttnArgs a{};
    a.early_trigger = g_tuning.early_trigger;
    a.q = (const uint16_t *)q;
    a.k = (const uint16_t *)k;
    a.v = (const uint16_t *)v;
    a.seq_lens = seq_lens;
    a.out = (uint16_t *)out;
    a.out_f32 = out_f32;
    a.part_m = (float *)(c.wsb + c.ws.part_m);
    a.part_l = (float *)(c.wsb + c.ws.part_l);
    a.part_o = (float *)(c.wsb + c.ws.part_o);
    a.tickets = (uint32_t *)(c.wsb + c.ws.tickets);
    a.status = (uint32_t *)(c.wsb + c.ws.status);
    a.Hq = c.shape.num_q_heads;
    a.Hkv = c.shape.num_kv_heads;
    a.Nmax = c.shape.max_seq_len;
    a.scale = c.scale;
    a.wait_limit_us = g_tuning.wait_limit_us;
    a.wait_test = g_tuning.wait_test;
    return a;
}

td_status check_layer_ptrs(const void *q, const void *k, const void *v, const void *out,
                           const float *out_f32)
{
    if (!q || !k || !v || !out)
        return TD_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16))
        return TD_ERR_INVALID_ARG;
    if (out_f32 && !aligned(out_f32, 16))
        return TD_ERR_INVALID_ARG;
    return TD_OK;
}

// Launches of one full(+select) layer; arguments already validated.  pdl: the
// attention kernel follows a kernel of the same call (programmatic dependent
// launch); the first kernel of a call is ordered by the stream alone.
// Coverage selection (tau >= 0): a per-row budget instead of top_k for every
// row; counts (optional) receives the number of positions kept per row.
struct Coverage {
    float tau = -1.0f;
    int32_t *counts = nullptr;
};

td_status run_full(const Ctx &c, const void *q, const void *k, const void *v,
                   const int32_t *seq_lens, int top_k, int32_t *idx_out, void *out,
                   float *out_f32, float *scores_out, cudaStream_t st, bool pdl,
                   Coverage cov = Coverage{}, int next_mode = -1)
{
    const bool select = top_k > 0;
    td::AttnArgs a = base_args(c, q, k, v, seq_lens, out, out_f32);
    a.scores = select ? (scores_out ? scores_out : (float *)(c.wsb + c.ws.scores)) : nullptr;
    a.hist = select ? (unsigned *)(c.wsb + c.ws.hist) : nullptr;
    a.prefetch = prefetch_for(c.G);
    // Measured on GB300 (graph steps): interleaved rounds keep a pair's CTAs
    // reading neighbouring rows at any moment; serving batch 1830 -> 1813 us
    // (tensor cores), 100K 1423 -> 1410 us and 10K 285 -> 283 us (CUDA cores,
    // register-streamed), 32K even (a read-only probe: grid-stride 6.9 TB/s
    // against 5.8 TB/s for one contiguous chunk per CTA at 4 CTAs per SM).
    a.interleave = g_tuning.full_interleave;
    plan_splits(c.shape, c.shape.max_seq_len, false, select, a.nsplit, a.chunk);
    const bool cluster = g_tuning.cluster && a.nsplit > 1 && a.nsplit <= td::kPortableClusterSplits;
    const cudaError_t le =
        mma_for(c.G) ? td::launch_attention_mma(c.G, false, select, mma_tokens_for(false), a,
                                                c.shape.batch, pdl, st)
                     : td::launch_attention(c.G, false, select, cluster,
                                            staged_for(c.shape, false, c.shape.max_seq_len), a,
                                            c.shape.batch, pdl, st);
    if (le != cudaSuccess)
        return TD_ERR_CUDA;
    if (select) {
        td::TopkArgs t{};
        t.scores = a.scores;
        t.hist = a.hist;
        t.seq_lens = seq_lens;
        t.idx = idx_out;
        t.status = a.status;
        t.Hkv = c.shape.num_kv_heads;
        t.Nmax = c.shape.max_seq_len;
        t.top_k = top_k;
        t.warp_select_max = g_tuning.topk_warp_max;
        if (cov.tau >= 0.0f) {
            td::CoverageArgs ca{};
            ca.scores = a.scores;
            ca.hist = a.hist;
            ca.seq_lens = seq_lens;
            ca.row_k = (int32_t *)(c.wsb + c.ws.row_k);
            ca.gcnt = (unsigned *)(c.wsb + c.ws.cov_cnt);
            ca.gmass = (float *)(c.wsb + c.ws.cov_mass);
            ca.Hkv = c.shape.num_kv_heads;
            ca.Nmax = c.shape.max_seq_len;
            ca.kcap = top_k;
            ca.tau = cov.tau;
            if (td::launch_coverage(ca, c.shape.batch, g_tuning.pdl != 0, st) != cudaSuccess)
                return TD_ERR_CUDA;
            t.row_k = ca.row_k;
            t.counts = cov.counts;
        }
        if (td::launch_topk(t, c.shape.batch, topk_threads_for(c.shape, top_k, next_mode),
                            topk_cluster_for(c.shape), g_tuning.pdl != 0 && g_tuning.topk_pdl != 0,
                            st) != cudaSuccess)
            return TD_ERR_CUDA;
    }
    return TD_OK;
}

// idx_dep: the kernel launched just before may have written `idx` (then the
// sparse kernel waits for it before reading the set).
// Stream-K plan of a tensor-core sparse launch (16 tokens per warp): whole
// waves of CTAs share the layer's B * Hkv * R rounds evenly, at most
// kMaxSparseChunk index entries per CTA; two rounds in flight per warp when
// the CTAs get 16 rounds or more.  a.nsplit becomes the partial stride: the
// largest number of CTAs that meet one (batch row, KV head).  False (plan
// unchanged) when the workspace's partials cannot hold them.
bool plan_stream_k(const Ctx &c, int top_k, td::AttnArgs &a, int &tokens)
{
    const long units = (long)c.shape.batch * c.shape.num_kv_heads;
    if (top_k < 1 || units > (1L << 16))
        return false;
    const long R = ceil_div(top_k, td::kTokPerRound);
    const long W = units * R;
    const long sms = device_sm_count();
    const long slots32 = sms * td::attention_mma_ctas_per_sm(c.G, true, false, 32);
    const bool db = W >= slots32 * 16;
    tokens = db ? 32 : 16;
    const long slots = db ? slots32 : sms * td::attention_mma_ctas_per_sm(c.G, true, false, 16);
    const long cap = td::kMaxSparseChunk / td::kTokPerRound;  // rounds one CTA stages
    const long waves = ceil_div(W, slots * cap);
    long P = slots * (waves > 0 ? waves : 1);
    if (P > W)
        P = W;
    long most = 1;  // CTAs meeting one (batch row, KV head); CTA of round y: ((y+1)P-1)/W
    for (long u = 0; u < units; ++u) {
        const long pf = ((u * R + 1) * P - 1) / W, pl = ((u + 1) * R * P - 1) / W;
        if (pl - pf + 1 > most)
            most = pl - pf + 1;
    }
    if (units * most > partial_slots(c.shape, top_k))
        return false;
    a.sk_ctas = (int)P;
    a.sk_units = (int)units;
    a.nsplit = (int)most;
    return true;
}

td_status run_sparse(const Ctx &c, const void *q, const void *k, const void *v,
                     const int32_t *seq_lens, const int32_t *idx, int top_k, void *out,
                     float *out_f32, cudaStream_t st, bool idx_dep, bool pdl)
{
    td::AttnArgs a = base_args(c, q, k, v, seq_lens, out, out_f32);
    a.idx = idx;
    a.top_k = top_k;
    a.idx_dep = idx_dep ? 1 : 0;
    plan_splits(c.shape, top_k, true, false, a.nsplit, a.chunk);
    const bool cluster = g_tuning.cluster && a.nsplit > 1 && a.nsplit <= td::kPortableClusterSplits;
    const int staged = staged_for(c.shape, true, top_k);
    int sk_tokens = 0;
    if (mma_for(c.G) && g_tuning.sparse_stream_k > 0 && plan_stream_k(c, top_k, a, sk_tokens)) {
        if (td::launch_attention_mma(c.G, true, false, sk_tokens, a, c.shape.batch, pdl, st) !=
            cudaSuccess)
            return TD_ERR_CUDA;
        return TD_OK;
    }
    if (!mma_for(c.G) && !cluster && staged == 2) {
        const long rows = (long)c.shape.batch * c.shape.num_kv_heads * c.shape.max_seq_len;
        if (!encode_row_map(&a.tma_k, k, rows) || !encode_row_map(&a.tma_v, v, rows))
            return TD_ERR_UNSUPPORTED_SHAPE;
        a.tma_rows = (int)rows;
    }
    const cudaError_t le =
        mma_for(c.G) ? td::launch_attention_mma(c.G, true, false,
                                                mma_tokens_for(true), a,
                                                c.shape.batch, pdl, st)
                     : td::launch_attention(c.G, true, false, cluster, staged, a,
                                            c.shape.batch, pdl, st);
    if (le != cudaSuccess)
        return TD_ERR_CUDA;
    return TD_OK;
}

td_status validate_step(const Ctx &c, int32_t num_layers, const int32_t *modes,
                        const void *const *q, const void *const *k_caches,
                        const void *const *v_caches, const int32_t *seq_lens, int32_t top_k,
                        const int32_t *idx_buf, int32_t idx_valid, void *const *outs,
                        float *const *outs_f32, const void *const *k_new,
                        const void *const *v_new)
{
    (void)c;
    if ((k_new == nullptr) != (v_new == nullptr))
        return TD_ERR_INVALID_ARG;
    if (num_layers < 0 || (num_layers > 0 && (!modes || !q || !k_caches || !v_caches || !outs)))
        return TD_ERR_INVALID_ARG;
    if (!seq_lens || !aligned(seq_lens, 4))
        return TD_ERR_INVALID_ARG;
    bool have_set = idx_valid != 0;
    bool uses_idx = false;
    for (int l = 0; l < num_layers; ++l) {
        const int m = modes[l];
        if (m != TD_MODE_FULL && m != TD_MODE_FULL_SELECT && m != TD_MODE_SPARSE)
            return TD_ERR_INVALID_ARG;
        td_status st = check_layer_ptrs(q[l], k_caches[l], v_caches[l], outs[l],
                                        outs_f32 ? outs_f32[l] : nullptr);
        if (st)
            return st;
        if (k_new && (!k_new[l] || !v_new[l] || !aligned(k_new[l], 16) || !aligned(v_new[l], 16)))
            return TD_ERR_INVALID_ARG;
        if (m == TD_MODE_FULL_SELECT) {
            if (top_k < 1)
                return TD_ERR_INVALID_ARG;
            have_set = true;
            uses_idx = true;
        } else if (m == TD_MODE_SPARSE) {
            if (top_k < 1)
                return TD_ERR_INVALID_ARG;
            if (!have_set)
                return TD_ERR_NO_SELECTION;
            uses_idx = true;
        }
    }
    if (uses_idx && (!idx_buf || !aligned(idx_buf, 4)))
        return TD_ERR_INVALID_ARG;
    return TD_OK;
}

// Host input/output of a captured step (td_plan_create_host), every layer's
// rows in one buffer per side.  With copy kernels (host_copy 1, the default,
// when both host buffers are mapped): the q rows by a kernel ahead of layer 0
// in the programmatic launch chain (layer 0's CTAs launch while it runs) --
// above 1 MiB only layer 0's, the rest by the copy engines on a side stream
// beside layer 0, which layer 1 waits for; the outputs of every 8 layers by
// the copy engines on the side stream once their last layer is done; the
// last two layers' by a kernel after the last layer, then the side stream is
// joined.  Copy engines only (host_copy 0, or unmapped buffers): one q copy
// before layer 0, the outputs of layers 0 .. L-2 once layer L-2 is done, the
// last layer's after it.  Measured on GB300 (graph steps, e2e against the
// same step on device buffers): copy kernels 100K 1398.9 / 1399.8 us, 32K
// 743.3 / 738.7, serving batch k = 1024 1787.6 / 1770.3, 10K 281.0 / 279.5;
// copy engines 1417.7, 760.2, 1850.5, 297.8 us.  Also measured: copy kernels
// with one output copy on the side stream after layer L-2 (1400.3, 746.6,
// 1843.1, 284.0 us: at 10K the copy is not hidden by the short last layer),
// all outputs by the tail kernel (1399.1, 749.8, 1861.9, 279.7 us), chunked
// outputs without the q split (1399.3, 743.6, 1816.6, 280.7 us).  One copy
// per layer costs 20-100 us a step, and a wait on a q copy before every layer
// breaks the programmatic launches between layers (32K +150 us).
struct StepIo {
    const void *q_host;
    void *q;
    void *outs;
    void *out_host;
    size_t layer_bytes;  // B * Hq * 128 * 2
    cudaStream_t stream;
    cudaEvent_t *ev;
    // device addresses of the two host buffers (page-locked host memory is
    // mapped into the device's address space): the copies run as kernels
    // when both are set and every buffer is 16-byte aligned
    const void *q_host_dev;
    void *out_host_dev;
    int mode;  // host_copy tuning at capture
};

constexpr size_t kSplitQBytes = size_t(1) << 20;  // q rows above this come in beside layer 0
constexpr int kOutChunkLayers = 8;                // layers per side-stream output copy

// Copies n 16-byte words between host and device memory, read or written by
// the SMs over the chip-to-chip link.  As a kernel it takes part in the
// step's programmatic launch chain: it waits for the kernel before it (when
// launched as a dependent), and lets the next one launch at once, so that
// kernel's CTAs request their first cache rows while the copy runs.
__global__ void __launch_bounds__(256) io_copy_kernel(const uint4 *__restrict__ src,
                                                      uint4 *__restrict__ dst, size_t n)
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    for (; i + 3 * stride < n; i += 4 * stride) {  // four loads in flight per thread
        const uint4 a = src[i], b = src[i + stride], c = src[i + 2 * stride],
                    d = src[i + 3 * stride];
        dst[i] = a;
        dst[i + stride] = b;
        dst[i + 2 * stride] = c;
        dst[i + 3 * stride] = d;
    }
    for (; i < n; i += stride)
        dst[i] = src[i];
}

cudaError_t launch_io_copy(const void *src, void *dst, size_t bytes, bool pdl, cudaStream_t st)
{
    const size_t n = bytes / 16;
    if (n == 0)
        return cudaSuccess;
    long grid = (long)ceil_div((long)n, 256);
    const long most = 4L * device_sm_count();
    if (grid > most)
        grid = most;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(256);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, io_copy_kernel, (const uint4 *)src, (uint4 *)dst, n);
}

td_status enqueue_step(const Ctx &c, int32_t num_layers, const int32_t *modes,
                       const void *const *q, const void *const *k_caches,
                       const void *const *v_caches, const int32_t *seq_lens, int32_t top_k,
                       int32_t *idx_buf, void *const *outs, float *const *outs_f32,
                       const void *const *k_new, const void *const *v_new, cudaStream_t st,
                       void *const *layer_events, const StepIo *io = nullptr)
{
    // KV append first: one launch per kAppendLayers layers writes every layer's
    // new rows; the first attention kernel is not overlapped with it.
    for (int l0 = 0; k_new && l0 < num_layers; l0 += td::kAppendLayers) {
        const int nl = num_layers - l0 < td::kAppendLayers ? num_layers - l0 : td::kAppendLayers;
        td::AppendBatch batch{};
        for (int j = 0; j < nl; ++j) {
            batch.k[j] = (uint16_t *)k_caches[l0 + j];
            batch.v[j] = (uint16_t *)v_caches[l0 + j];
            batch.k_new[j] = (const uint16_t *)k_new[l0 + j];
            batch.v_new[j] = (const uint16_t *)v_new[l0 + j];
        }
        if (td::launch_kv_append(batch, nl, seq_lens, c.shape.batch, c.shape.num_kv_heads,
                                 c.shape.max_seq_len, st) != cudaSuccess)
            return TD_ERR_CUDA;
    }
    // Host rows (see StepIo): which layers' outputs the tail copy takes, how
    // many layers each side-stream output copy takes, and whether the q rows
    // of layers 1 .. L-1 come in on the side stream beside layer 0.
    const bool io_kernels = io && io->mode > 0 && io->q_host_dev && io->out_host_dev;
    const int L = num_layers;
    const size_t lb = io ? io->layer_bytes : 0;
    int tail_from = L - 1, chunk = L;
    bool q_split = false;
    if (io_kernels) {
        tail_from = L >= 2 ? L - 2 : 0;
        chunk = kOutChunkLayers;
        q_split = L >= 2 && lb * L > kSplitQBytes;
    }
    if (io) {
        if (q_split) {
            if (cudaEventRecord(io->ev[0], st) != cudaSuccess ||
                cudaStreamWaitEvent(io->stream, io->ev[0], 0) != cudaSuccess ||
                cudaMemcpyAsync((char *)io->q + lb, (const char *)io->q_host + lb, lb * (L - 1),
                                cudaMemcpyHostToDevice, io->stream) != cudaSuccess ||
                cudaEventRecord(io->ev[1], io->stream) != cudaSuccess ||
                launch_io_copy(io->q_host_dev, io->q, lb, false, st) != cudaSuccess)
                return TD_ERR_CUDA;
        } else if ((io_kernels ? launch_io_copy(io->q_host_dev, io->q, lb * L, false, st)
                               : cudaMemcpyAsync(io->q, io->q_host, lb * L, cudaMemcpyHostToDevice,
                                                 st)) != cudaSuccess) {
            return TD_ERR_CUDA;
        }
    }
    int side_from = 0, n_side = 0;
    bool side_used = q_split;
    for (int l = 0; l < num_layers; ++l) {
        // the first kernel waits for what precedes it, except a copy kernel
        const bool pdl = (l > 0 || io_kernels) && g_tuning.pdl;
        if (q_split && l == 1 && cudaStreamWaitEvent(st, io->ev[1], 0) != cudaSuccess)
            return TD_ERR_CUDA;
        if (layer_events && layer_events[l] &&
            cudaEventRecord((cudaEvent_t)layer_events[l], st) != cudaSuccess)
            return TD_ERR_CUDA;
        float *of = outs_f32 ? outs_f32[l] : nullptr;
        td_status r;
        switch (modes[l]) {
        case TD_MODE_FULL:
            r = run_full(c, q[l], k_caches[l], v_caches[l], seq_lens, 0, nullptr, outs[l], of,
                         nullptr, st, pdl);
            break;
        case TD_MODE_FULL_SELECT:
            r = run_full(c, q[l], k_caches[l], v_caches[l], seq_lens, top_k, idx_buf,
                         outs[l], of, nullptr, st, pdl, Coverage{},
                         l + 1 < num_layers ? modes[l + 1] : -1);
            break;
        default:
            r = run_sparse(c, q[l], k_caches[l], v_caches[l], seq_lens, idx_buf, top_k,
                           outs[l], of, st, l == 0 || modes[l - 1] == TD_MODE_FULL_SELECT, pdl);
            break;
        }
        if (r)
            return r;
        // host outputs of layers side_from .. l on the side stream once layer l is done
        if (io && l < tail_from && (l + 1 - side_from == chunk || l == tail_from - 1)) {
            cudaEvent_t e = io->ev[3 + n_side++];
            if (cudaEventRecord(e, st) != cudaSuccess ||
                cudaStreamWaitEvent(io->stream, e, 0) != cudaSuccess ||
                cudaMemcpyAsync((char *)io->out_host + lb * side_from,
                                (const char *)io->outs + lb * side_from, lb * (l + 1 - side_from),
                                cudaMemcpyDeviceToHost, io->stream) != cudaSuccess)
                return TD_ERR_CUDA;
            side_from = l + 1;
            side_used = true;
        }
    }
    // the remaining layers' outputs, then join the side stream
    if (io) {
        const size_t first = lb * tail_from, bytes = lb * (L - tail_from);
        const cudaError_t e =
            io_kernels ? launch_io_copy((const char *)io->outs + first,
                                        (char *)io->out_host_dev + first, bytes, g_tuning.pdl, st)
                       : cudaMemcpyAsync((char *)io->out_host + first,
                                         (const char *)io->outs + first, bytes,
                                         cudaMemcpyDeviceToHost, st);
        if (e != cudaSuccess ||
            (side_used && (cudaEventRecord(io->ev[2], io->stream) != cudaSuccess ||
                           cudaStreamWaitEvent(st, io->ev[2], 0) != cudaSuccess)))
            return TD_ERR_CUDA;
    }
    if (layer_events && layer_events[num_layers] &&
        cudaEventRecord((cudaEvent_t)layer_events[num_layers], st) != cudaSuccess)
        return TD_ERR_CUDA;
    return TD_OK;
}

}  // namespace

struct td_plan {
    cudaGraph_t graph = nullptr;
    cudaGraphExec_t exec = nullptr;
};

namespace {

// Host memory the copy engines can read and write asynchronously.
bool page_locked(const void *p)
{
    if (!p)
        return false;
    cudaPointerAttributes attr{};
    if (cudaPointerGetAttributes(&attr, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return attr.type == cudaMemoryTypeHost;
}

// Captures a step (optionally with host q in and outputs out) into a graph.
td_status create_plan(td_plan **plan, const td_shape *shape, int32_t num_layers,
                      const int32_t *modes, const void *const *q, const void *const *k_caches,
                      const void *const *v_caches, const void *const *k_new,
                      const void *const *v_new, const int32_t *seq_lens, int32_t top_k,
                      int32_t *idx_buf, int32_t idx_valid, void *const *outs,
                      float *const *outs_f32, void *ws, size_t ws_bytes,
                      const StepIo *host = nullptr)
{
    if (!plan)
        return TD_ERR_INVALID_ARG;
    *plan = nullptr;
    Ctx c;
    td_status st = make_ctx(shape, top_k, ws, ws_bytes, c);
    if (st)
        return st;
    st = validate_step(c, num_layers, modes, q, k_caches, v_caches, seq_lens, top_k, idx_buf,
                       idx_valid, outs, outs_f32, k_new, v_new);
    if (st)
        return st;
    td_plan *p = new (std::nothrow) td_plan();
    if (!p)
        return TD_ERR_INVALID_ARG;
    const bool host_io = host != nullptr;
    std::vector<cudaEvent_t> ev(host_io ? 3 + num_layers : 0, nullptr);
    cudaStream_t cap = nullptr, side = nullptr;
    bool ok = cudaStreamCreateWithFlags(&cap, cudaStreamNonBlocking) == cudaSuccess;
    if (ok && host_io) {
        ok = cudaStreamCreateWithFlags(&side, cudaStreamNonBlocking) == cudaSuccess;
        for (size_t i = 0; ok && i < ev.size(); ++i)
            ok = cudaEventCreateWithFlags(&ev[i], cudaEventDisableTiming) == cudaSuccess;
    }
    if (!ok) {
        st = TD_ERR_CUDA;
    } else if (cudaStreamBeginCapture(cap, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
        st = TD_ERR_CUDA;
    } else {
        StepIo io = host ? *host : StepIo{};
        io.stream = side;
        io.ev = ev.data();
        td_status enq = enqueue_step(c, num_layers, modes, q, k_caches, v_caches, seq_lens,
                                     top_k, idx_buf, outs, outs_f32, k_new, v_new, cap, nullptr,
                                     host_io ? &io : nullptr);
        cudaGraph_t graph = nullptr;
        const cudaError_t end = cudaStreamEndCapture(cap, &graph);
        if (enq != TD_OK || end != cudaSuccess) {
            st = enq != TD_OK ? enq : TD_ERR_CUDA;
            if (graph)
                cudaGraphDestroy(graph);
            cudaGetLastError();
        } else {
            p->graph = graph;
            if (cudaGraphInstantiate(&p->exec, graph, 0) != cudaSuccess)
                st = TD_ERR_CUDA;
        }
    }
    for (cudaEvent_t e : ev)
        if (e)
            cudaEventDestroy(e);
    if (side)
        cudaStreamDestroy(side);
    if (cap)
        cudaStreamDestroy(cap);
    if (st) {
        td_plan_destroy(p);
        return st;
    }
    *plan = p;
    return TD_OK;
}

}  // namespace

extern "C" {

const char *td_status_string(td_status status)
{
    switch (status) {
    case TD_OK: return "TD_OK";
    case TD_ERR_INVALID_ARG: return "TD_ERR_INVALID_ARG";
    case TD_ERR_UNSUPPORTED_SHAPE: return "TD_ERR_UNSUPPORTED_SHAPE";
    case TD_ERR_NO_SELECTION: return "TD_ERR_NO_SELECTION";
    case TD_ERR_WORKSPACE_TOO_SMALL: return "TD_ERR_WORKSPACE_TOO_SMALL";
    case TD_ERR_CUDA: return "TD_ERR_CUDA";
    }
    return "TD_ERR_UNKNOWN";
}

size_t td_workspace_size(const td_shape *shape, int32_t top_k)
{
    if (check_shape(shape) != TD_OK || top_k < 0 || top_k > shape->max_seq_len ||
        top_k > td::kMaxTopK)
        return 0;
    return ws_layout(*shape, top_k).total;
}

td_status td_workspace_init(void *ws, size_t ws_bytes, void *stream)
{
    if (!ws || !aligned(ws, kAlign) || ws_bytes < kAlign)
        return TD_ERR_INVALID_ARG;
    if (cudaMemsetAsync(ws, 0, ws_bytes, (cudaStream_t)stream) != cudaSuccess)
        return TD_ERR_CUDA;
    return TD_OK;
}

td_status td_workspace_status(void *ws, size_t ws_bytes, uint32_t *flags, void *stream)
{
    if (!ws || !flags || !aligned(ws, kAlign) || ws_bytes < kAlign)
        return TD_ERR_INVALID_ARG;
    cudaStream_t st = (cudaStream_t)stream;
    uint32_t host = 0;
    if (cudaMemcpyAsync(&host, ws, sizeof host, cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaMemsetAsync(ws, 0, sizeof(uint32_t), st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
        return TD_ERR_CUDA;
    *flags = host;
    return TD_OK;
}

td_status td_full_attn_select(const td_shape *shape, const void *q, const void *k_cache,
                              const void *v_cache, const int32_t *seq_lens, int32_t top_k,
                              int32_t *idx_out, void *out, float *out_f32, float *scores_out,
                              void *ws, size_t ws_bytes, void *stream)
{
    Ctx c;
    td_status st = make_ctx(shape, top_k, ws, ws_bytes, c);
    if (st)
        return st;
    st = check_layer_ptrs(q, k_cache, v_cache, out, out_f32);
    if (st)
        return st;
    if (!seq_lens || !aligned(seq_lens, 4))
        return TD_ERR_INVALID_ARG;
    if (top_k > 0 && (!idx_out || !aligned(idx_out, 4)))
        return TD_ERR_INVALID_ARG;
    if (scores_out && !aligned(scores_out, 4))
        return TD_ERR_INVALID_ARG;
    return run_full(c, q, k_cache, v_cache, seq_lens, top_k, idx_out, out, out_f32,
                    top_k > 0 ? scores_out : nullptr, (cudaStream_t)stream, false);
}

td_status td_full_attn_select_coverage(const td_shape *shape, const void *q, const void *k_cache,
                                       const void *v_cache, const int32_t *seq_lens, float tau,
                                       int32_t k_max, int32_t *idx_out, int32_t *counts_out,
                                       void *out, float *out_f32, float *scores_out, void *ws,
                                       size_t ws_bytes, void *stream)
{
    Ctx c;
    td_status st = make_ctx(shape, k_max, ws, ws_bytes, c);
    if (st)
        return st;
    st = check_layer_ptrs(q, k_cache, v_cache, out, out_f32);
    if (st)
        return st;
    if (!(tau >= 0.0f && tau < 1.0f) || k_max < 1 || !idx_out || !aligned(idx_out, 4) ||
        !seq_lens || !aligned(seq_lens, 4) || (counts_out && !aligned(counts_out, 4)) ||
        (scores_out && !aligned(scores_out, 4)))
        return TD_ERR_INVALID_ARG;
    Coverage cov;
    cov.tau = tau;
    cov.counts = counts_out;
    return run_full(c, q, k_cache, v_cache, seq_lens, k_max, idx_out, out, out_f32,
                    scores_out, (cudaStream_t)stream, false, cov);
}

td_status td_topk_select(const td_shape *shape, const float *scores, const int32_t *seq_lens,
                         int32_t top_k, int32_t *idx_out, void *ws, size_t ws_bytes,
                         void *stream)
{
    Ctx c;
    td_status st = make_ctx(shape, top_k, ws, ws_bytes, c);
    if (st)
        return st;
    if (top_k < 1 || !scores || !aligned(scores, 4) || !seq_lens || !aligned(seq_lens, 4) ||
        !idx_out || !aligned(idx_out, 4))
        return TD_ERR_INVALID_ARG;
    td::TopkArgs t{};
    t.scores = scores;
    t.seq_lens = seq_lens;
    t.idx = idx_out;
    t.status = (uint32_t *)(c.wsb + c.ws.status);
    t.Hkv = c.shape.num_kv_heads;
    t.Nmax = c.shape.max_seq_len;
    t.top_k = top_k;
    t.warp_select_max = g_tuning.topk_warp_max;
    if (td::launch_topk(t, c.shape.batch, topk_threads_for(c.shape, top_k, -1),
                        topk_cluster_for(c.shape), false, (cudaStream_t)stream) != cudaSuccess)
        return TD_ERR_CUDA;
    return TD_OK;
}

td_status td_probe_layer_reads(const td_shape *shape, const void *k_cache, const void *v_cache,
                               const int32_t *seq_lens, const int32_t *idx, int32_t top_k,
                               uint32_t *sink, int32_t sink_words, void *stream)
{
    td_status st = check_shape(shape);
    if (st)
        return st;
    const bool sparse = idx != nullptr;
    if (!k_cache || !v_cache || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !seq_lens ||
        !aligned(seq_lens, 4) || !sink || !aligned(sink, 4) || sink_words < 1 ||
        (sparse && (!aligned(idx, 4) || top_k < 1 || top_k > shape->max_seq_len)))
        return TD_ERR_INVALID_ARG;
    td::ProbeArgs a{};
    a.k = (const uint16_t *)k_cache;
    a.v = (const uint16_t *)v_cache;
    a.seq_lens = seq_lens;
    a.idx = idx;
    a.sink = sink;
    a.sink_words = sink_words;
    a.Hkv = shape->num_kv_heads;
    a.Nmax = shape->max_seq_len;
    a.top_k = sparse ? top_k : 0;
    plan_splits(*shape, sparse ? top_k : shape->max_seq_len, sparse, false, a.nsplit, a.chunk);
    if (td::launch_probe_reads(a, shape->batch, (cudaStream_t)stream) != cudaSuccess)
        return TD_ERR_CUDA;
    return TD_OK;
}

td_status td_index_overlap(const td_shape *shape, const int32_t *idx_a, const int32_t *idx_b,
                           int32_t top_k, int32_t *counts, void *stream)
{
    td_status st = check_shape(shape);
    if (st)
        return st;
    if (top_k < 1 || top_k > td::kMaxTopK || !idx_a || !aligned(idx_a, 4) || !idx_b ||
        !aligned(idx_b, 4) || !counts || !aligned(counts, 4))
        return TD_ERR_INVALID_ARG;
    const int rows = shape->batch * shape->num_kv_heads;
    if (td::launch_index_overlap(idx_a, idx_b, rows, top_k, counts, (cudaStream_t)stream) !=
        cudaSuccess)
        return TD_ERR_CUDA;
    return TD_OK;
}

td_status td_sparse_attn(const td_shape *shape, const void *q, const void *k_cache,
                         const void *v_cache, const int32_t *seq_lens, const int32_t *idx,
                         int32_t top_k, void *out, float *out_f32, void *ws, size_t ws_bytes,
                         void *stream)
{
    Ctx c;
    td_status st = make_ctx(shape, top_k, ws, ws_bytes, c);
    if (st)
        return st;
    st = check_layer_ptrs(q, k_cache, v_cache, out, out_f32);
    if (st)
        return st;
    if (top_k < 1 || !idx || !aligned(idx, 4) || !seq_lens || !aligned(seq_lens, 4))
        return TD_ERR_INVALID_ARG;
    return run_sparse(c, q, k_cache, v_cache, seq_lens, idx, top_k, out, out_f32,
                      (cudaStream_t)stream, true, false);
}

td_status td_decode_step(const td_shape *shape, int32_t num_layers, const int32_t *modes,
                         const void *const *q, const void *const *k_caches,
                         const void *const *v_caches, const int32_t *seq_lens, int32_t top_k,
                         int32_t *idx_buf, int32_t idx_valid, void *const *outs,
                         float *const *outs_f32, void *ws, size_t ws_bytes, void *stream,
                         void *const *layer_events)
{
    return td_decode_step_append(shape, num_layers, modes, q, k_caches, v_caches, nullptr,
                                 nullptr, seq_lens, top_k, idx_buf, idx_valid, outs, outs_f32, ws,
                                 ws_bytes, stream, layer_events);
}

td_status td_decode_step_append(const td_shape *shape, int32_t num_layers, const int32_t *modes,
                                const void *const *q, const void *const *k_caches,
                                const void *const *v_caches, const void *const *k_new,
                                const void *const *v_new, const int32_t *seq_lens,
                                int32_t top_k, int32_t *idx_buf, int32_t idx_valid,
                                void *const *outs, float *const *outs_f32, void *ws,
                                size_t ws_bytes, void *stream, void *const *layer_events)
{
    Ctx c;
    td_status st = make_ctx(shape, top_k, ws, ws_bytes, c);
    if (st)
        return st;
    st = validate_step(c, num_layers, modes, q, k_caches, v_caches, seq_lens, top_k, idx_buf,
                       idx_valid, outs, outs_f32, k_new, v_new);
    if (st)
        return st;
    return enqueue_step(c, num_layers, modes, q, k_caches, v_caches, seq_lens, top_k, idx_buf,
                        outs, outs_f32, k_new, v_new, (cudaStream_t)stream, layer_events);
}

td_status td_kv_append(const td_shape *shape, void *k_cache, void *v_cache, const void *k_new,
                       const void *v_new, const int32_t *seq_lens, void *stream)
{
    td_status st = check_shape(shape);
    if (st)
        return st;
    if (!k_cache || !v_cache || !k_new || !v_new || !aligned(k_cache, 16) ||
        !aligned(v_cache, 16) || !aligned(k_new, 16) || !aligned(v_new, 16) || !seq_lens ||
        !aligned(seq_lens, 4))
        return TD_ERR_INVALID_ARG;
    td::AppendBatch batch{};
    batch.k[0] = (uint16_t *)k_cache;
    batch.v[0] = (uint16_t *)v_cache;
    batch.k_new[0] = (const uint16_t *)k_new;
    batch.v_new[0] = (const uint16_t *)v_new;
    if (td::launch_kv_append(batch, 1, seq_lens, shape->batch, shape->num_kv_heads,
                             shape->max_seq_len, (cudaStream_t)stream) != cudaSuccess)
        return TD_ERR_CUDA;
    return TD_OK;
}

td_status td_plan_create(td_plan **plan, const td_shape *shape, int32_t num_layers,
                         const int32_t *modes, const void *const *q,
                         const void *const *k_caches, const void *const *v_caches,
                         const int32_t *seq_lens, int32_t top_k, int32_t *idx_buf,
                         int32_t idx_valid, void *const *outs, float *const *outs_f32, void *ws,
                         size_t ws_bytes)
{
    return td_plan_create_append(plan, shape, num_layers, modes, q, k_caches, v_caches, nullptr,
                                 nullptr, seq_lens, top_k, idx_buf, idx_valid, outs, outs_f32, ws,
                                 ws_bytes);
}

td_status td_plan_create_append(td_plan **plan, const td_shape *shape, int32_t num_layers,
                                const int32_t *modes, const void *const *q,
                                const void *const *k_caches, const void *const *v_caches,
                                const void *const *k_new, const void *const *v_new,
                                const int32_t *seq_lens, int32_t top_k, int32_t *idx_buf,
                                int32_t idx_valid, void *const *outs, float *const *outs_f32,
                                void *ws, size_t ws_bytes)
{
    return create_plan(plan, shape, num_layers, modes, q, k_caches, v_caches, k_new, v_new,
                       seq_lens, top_k, idx_buf, idx_valid, outs, outs_f32, ws, ws_bytes);
}

td_status td_plan_create_host(td_plan **plan, const td_shape *shape, int32_t num_layers,
                              const int32_t *modes, const void *q_host, void *q,
                              const void *const *k_caches, const void *const *v_caches,
                              const int32_t *seq_lens, int32_t top_k, int32_t *idx_buf,
                              int32_t idx_valid, void *outs, float *const *outs_f32,
                              void *out_host, void *ws, size_t ws_bytes)
{
    if (!plan)
        return TD_ERR_INVALID_ARG;
    *plan = nullptr;
    if (check_shape(shape) != TD_OK || num_layers < 1 || !q || !outs)
        return TD_ERR_INVALID_ARG;
    if (!page_locked(q_host) || !page_locked(out_host))
        return TD_ERR_INVALID_ARG;
    StepIo io{};
    io.q_host = q_host;
    io.q = q;
    io.outs = outs;
    io.out_host = out_host;
    io.layer_bytes = (size_t)shape->batch * shape->num_q_heads * kHeadDim * sizeof(uint16_t);
    io.mode = g_tuning.host_copy;
    void *dq = nullptr, *dout = nullptr;
    if (io.mode > 0 && aligned(q_host, 16) && aligned(out_host, 16) && aligned(q, 16) &&
        aligned(outs, 16) &&
        cudaHostGetDevicePointer(&dq, const_cast<void *>(q_host), 0) == cudaSuccess &&
        cudaHostGetDevicePointer(&dout, out_host, 0) == cudaSuccess) {
        io.q_host_dev = dq;
        io.out_host_dev = dout;
    } else {
        cudaGetLastError();  // not mapped: the copy engines move the rows
    }
    std::vector<const void *> qs(num_layers);
    std::vector<void *> os(num_layers);
    for (int l = 0; l < num_layers; ++l) {
        qs[l] = (const char *)q + io.layer_bytes * l;
        os[l] = (char *)outs + io.layer_bytes * l;
    }
    return create_plan(plan, shape, num_layers, modes, qs.data(), k_caches, v_caches, nullptr,
                       nullptr, seq_lens, top_k, idx_buf, idx_valid, os.data(), outs_f32, ws,
                       ws_bytes, &io);
}

td_status td_plan_launch(td_plan *plan, void *stream)
{
    if (!plan || !plan->exec)
        return TD_ERR_INVALID_ARG;
    if (cudaGraphLaunch(plan->exec, (cudaStream_t)stream) != cudaSuccess)
        return TD_ERR_CUDA;
    return TD_OK;
}

void td_plan_destroy(td_plan *plan)
{
    if (!plan)
        return;
    if (plan->exec)
        cudaGraphExecDestroy(plan->exec);
    if (plan->graph)
        cudaGraphDestroy(plan->graph);
    delete plan;
}

td_status td_set_tuning(const char *key, int32_t value)
{
    if (!key)
        return TD_ERR_INVALID_ARG;
    if (!strcmp(key, "full_ctas_per_sm"))
        g_tuning.full_ctas_per_sm = value > 0 ? value : kDefaultTuning.full_ctas_per_sm;
    else if (!strcmp(key, "sparse_ctas_per_sm"))
        g_tuning.sparse_ctas_per_sm = value > 0 ? value : kDefaultTuning.sparse_ctas_per_sm;
    else if (!strcmp(key, "full_waves"))
        g_tuning.full_waves = value > 0 ? value : kDefaultTuning.full_waves;
    else if (!strcmp(key, "sparse_waves"))
        g_tuning.sparse_waves = value > 0 ? value : kDefaultTuning.sparse_waves;
    else if (!strcmp(key, "sparse_splits"))
        g_tuning.sparse_splits = (value > 0 && value <= td::kMaxSplits) ? value
                                                                       : kDefaultTuning.sparse_splits;
    else if (!strcmp(key, "cluster"))
        g_tuning.cluster = value > 0 ? 1 : 0;
    else if (!strcmp(key, "full_staged"))
        g_tuning.full_staged = value > 0 ? 1 : (value == 0 ? 0 : kDefaultTuning.full_staged);  // <0: auto
    else if (!strcmp(key, "sparse_staged"))
        g_tuning.sparse_staged = (value >= 0 && value <= 2) ? value : kDefaultTuning.sparse_staged;
    else if (!strcmp(key, "mma"))
        g_tuning.mma = value > 0 ? 1 : (value == 0 ? 0 : kDefaultTuning.mma);
    else if (!strcmp(key, "full_prefetch"))
        g_tuning.full_prefetch = (value >= 0 && value <= 4) ? value : kDefaultTuning.full_prefetch;
    else if (!strcmp(key, "topk_warp_max"))
        g_tuning.topk_warp_max = value > 0 ? value : kDefaultTuning.topk_warp_max;
    else if (!strcmp(key, "pdl"))
        g_tuning.pdl = value != 0 ? 1 : 0;
    else if (!strcmp(key, "topk_pdl"))
        g_tuning.topk_pdl = value != 0 ? 1 : 0;
    else if (!strcmp(key, "sparse_stream_k"))
        g_tuning.sparse_stream_k = value > 0 ? 1 : (value == 0 ? 0 : kDefaultTuning.sparse_stream_k);
    else if (!strcmp(key, "mma_full_tokens"))
        g_tuning.mma_full_tokens =
            (value == 8 || value == 16 || value == 32) ? value : kDefaultTuning.mma_full_tokens;
    else if (!strcmp(key, "mma_sparse_tokens"))
        g_tuning.mma_sparse_tokens =
            (value == 8 || value == 16 || value == 32 || value == 64)
                ? value
                : kDefaultTuning.mma_sparse_tokens;
    else if (!strcmp(key, "full_interleave"))
        g_tuning.full_interleave = value > 0 ? 1 : (value == 0 ? 0 : kDefaultTuning.full_interleave);
    else if (!strcmp(key, "early_trigger"))
        g_tuning.early_trigger = (value >= 0 && value <= 64) ? value : kDefaultTuning.early_trigger;
    else if (!strcmp(key, "host_copy"))
        g_tuning.host_copy = (value == 0 || value == 1) ? value : kDefaultTuning.host_copy;
    else if (!strcmp(key, "wait_limit_us"))
        g_tuning.wait_limit_us = value > 0 ? value : kDefaultTuning.wait_limit_us;
    else if (!strcmp(key, "wait_test"))
        g_tuning.wait_test = value > 0 ? 1 : 0;
    else if (!strcmp(key, "topk_cluster"))
        g_tuning.topk_cluster = (value == 1 || value == 2 || value == 4 || value == 8)
                                    ? value
                                    : kDefaultTuning.topk_cluster;
    else if (!strcmp(key, "topk_threads"))
        g_tuning.topk_threads = (value == 512 || value == 1024) ? value : 0;
    else if (!strcmp(key, "attn_carveout"))
        td::set_attention_carveout(value >= 0 && value <= 100 ? value : -1);
    else if (!strcmp(key, "max_splits"))
        g_tuning.max_splits = (value > 0 && value <= td::kMaxSplits) ? value : td::kMaxSplits;
    else
        return TD_ERR_INVALID_ARG;
    return TD_OK;
}

const char *td_kernel_name(const td_shape *shape, int32_t top_k, int32_t sparse)
{
    if (check_shape(shape) != TD_OK || top_k < 0 || top_k > shape->max_seq_len)
        return "invalid shape";
    const int G = shape->num_q_heads / shape->num_kv_heads;
    const bool sp = sparse != 0;
    int nsplit = 0, chunk = 0;
    const long n_total = sp ? top_k : shape->max_seq_len;
    plan_splits(*shape, n_total, sp, !sp && top_k > 0, nsplit, chunk);
    if (mma_for(G)) {
        if (sp && g_tuning.sparse_stream_k > 0)
            return "attention_mma16_kernel (tensor cores, 16 tokens per warp, stream-K partition)";
        const int t = mma_tokens_for(sp);
        return t == 64   ? "attention_mma_ring_kernel (tensor cores, rounds staged in shared memory)"
               : t == 32 ? "attention_mma16_kernel (tensor cores, 16 tokens per warp, two rounds in flight)"
               : t == 16 ? "attention_mma16_kernel (tensor cores, 16 tokens per warp)"
                         : "attention_mma_kernel (tensor cores, 8 tokens per warp)";
    }
    if (g_tuning.cluster && nsplit > 1 && nsplit <= td::kPortableClusterSplits)
        return "attention_kernel (CUDA cores, register-streamed, cluster split merge)";
    switch (staged_for(*shape, sp, n_total)) {
    case 2: return "attention_kernel (CUDA cores, TMA row gathers into shared-memory stages)";
    case 1: return sp ? "attention_kernel (CUDA cores, cp.async rows into shared-memory stages)"
                      : "attention_kernel (CUDA cores, bulk copies into shared-memory stages)";
    default: return "attention_kernel (CUDA cores, register-streamed)";
    }
}

int32_t td_query_splits(const td_shape *shape, int32_t top_k, int32_t sparse)
{
    if (check_shape(shape) != TD_OK)
        return 0;
    int nsplit = 0, chunk = 0;
    plan_splits(*shape, sparse ? top_k : shape->max_seq_len, sparse != 0, !sparse && top_k > 0,
                nsplit, chunk);
    return nsplit;
}

}  // extern "C"
