// td_noalloc.cu -- td_sparse_attn_noalloc: the sparse (PPSA) attention layer
// for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc or hand the library a workspace: code
// that runs inside a host framework which owns all device memory through its
// own arena and forbids raw allocations, real-time paths that must not enter
// the driver's allocator (it can synchronise the device and has unbounded
// latency), and plugins loaded into a process whose memory budget is fixed
// before they run.  For them this entry point keeps its scratch (split
// partials, arrival tickets, status word) in one fixed array of
// TD_NOALLOC_SCRATCH_BYTES bytes that lives in the library's device image.
// Every GPU that loads the library holds that array until the process exits.
//
// Set-up: the first call on a device (with that device current) looks the
// array's device address up with cudaGetSymbolAddress and caches it per
// device, keyed on the CUDA context current at the time: a call that finds
// another context current (after cudaDeviceReset, or a driver-API context of
// the caller's) looks the address up again.  Make the first call in each
// context before any stream capture begins.
// Every call shares the one array per device, and it keeps what the last call
// left there: each call clears the tickets and status word (cudaMemsetAsync on
// its stream) before its kernel runs.  Calls whose kernels overlap on the GPU
// (different streams, or concurrent host threads) race on the array; order
// them on one stream.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <mutex>

#include "../../include/td.h"
#include "td_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[TD_NOALLOC_SCRATCH_BYTES];

constexpr size_t kNaAlign = 256;
constexpr int kMaxDevices = 64;
constexpr int kEntriesPerCta = 256;  // target index entries per CTA
constexpr int kMaxNoallocSplits = 64;
constexpr int kMmaSparseTokens = 8;  // tensor-core sparse kernel variant (tokens per warp per round)

inline size_t na_align(size_t x) { return (x + kNaAlign - 1) & ~(kNaAlign - 1); }
inline bool na_aligned(const void *p, size_t a) { return ((uintptr_t)p % a) == 0; }

std::mutex g_mu;
struct ScratchAddr {
    void *ctx;   // context the address was looked up in
    void *addr;  // device address of g_noalloc_scratch there
};
ScratchAddr g_scratch[kMaxDevices] = {};

// cuCtxGetCurrent, reached through the runtime (the library does not link the
// driver library itself); null if the driver does not provide it.
typedef int (*CtxGetCurrentFn)(void **);
CtxGetCurrentFn ctx_get_current()
{
    static CtxGetCurrentFn fn = [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            p = nullptr;
        return (CtxGetCurrentFn)p;
    }();
    return fn;
}

void *current_ctx()
{
    void *ctx = nullptr;
    if (CtxGetCurrentFn fn = ctx_get_current())
        if (fn(&ctx) != 0)
            ctx = nullptr;
    return ctx;
}

// Device address of the scratch array in the current context (cached per
// device and context).
td_status scratch_address(void **out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return TD_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    void *ctx = current_ctx();
    if (!g_scratch[dev].addr || !ctx || g_scratch[dev].ctx != ctx) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p)
            return TD_ERR_CUDA;
        g_scratch[dev].addr = p;
        g_scratch[dev].ctx = current_ctx();  // current now, if it was not before the lookup
    }
    *out = g_scratch[dev].addr;
    return TD_OK;
}

struct NaLayout {
    size_t status, tickets, part_m, part_l, part_o, total;
};

// With one split a CTA writes its (batch row, KV head)'s output itself, so
// the layout holds no partials then.
NaLayout na_layout(size_t units, int nsplit, int G)
{
    NaLayout L{};
    size_t off = 0;
    L.status = off;
    off = na_align(off + sizeof(uint32_t));
    L.tickets = off;
    off = na_align(off + units * sizeof(uint32_t));
    const size_t slots = nsplit > 1 ? units * (size_t)nsplit * (size_t)G : 0;
    L.part_m = off;
    off = na_align(off + slots * sizeof(float));
    L.part_l = off;
    off = na_align(off + slots * sizeof(float));
    L.part_o = off;
    off = na_align(off + slots * td::kHeadDim * sizeof(float));
    L.total = off;
    return L;
}

}  // namespace

extern "C" td_status td_sparse_attn_noalloc(const td_shape *shape, const void *q,
                                            const void *k_cache, const void *v_cache,
                                            const int32_t *seq_lens, const int32_t *idx,
                                            int32_t top_k, void *out, float *out_f32,
                                            void *stream)
{
    if (!shape)
        return TD_ERR_INVALID_ARG;
    const td_shape s = *shape;
    if (s.batch < 1 || s.num_q_heads < 1 || s.num_kv_heads < 1 || s.max_seq_len < 1 ||
        s.num_q_heads % s.num_kv_heads || !isfinite(s.scale) || s.scale < 0.0f)
        return TD_ERR_INVALID_ARG;
    const int G = s.num_q_heads / s.num_kv_heads;
    if (s.head_dim != td::kHeadDim || (G != 1 && G != 2 && G != 4 && G != 8) ||
        s.batch > 65535 || s.num_kv_heads > 65535)
        return TD_ERR_UNSUPPORTED_SHAPE;
    if (top_k < 1 || top_k > s.max_seq_len)
        return TD_ERR_INVALID_ARG;
    if (!q || !k_cache || !v_cache || !out || !idx || !seq_lens)
        return TD_ERR_INVALID_ARG;
    if (!na_aligned(q, 16) || !na_aligned(k_cache, 16) || !na_aligned(v_cache, 16) ||
        !na_aligned(out, 16) || (out_f32 && !na_aligned(out_f32, 16)) || !na_aligned(idx, 4) ||
        !na_aligned(seq_lens, 4))
        return TD_ERR_INVALID_ARG;

    // Splits: about kEntriesPerCta entries per CTA, then as few as the fixed
    // scratch needs; a CTA stages at most kMaxSparseChunk entries.
    const size_t units = (size_t)s.batch * s.num_kv_heads;
    int nsplit = (top_k + kEntriesPerCta - 1) / kEntriesPerCta;
    if (nsplit > kMaxNoallocSplits)
        nsplit = kMaxNoallocSplits;
    if (nsplit < 1)
        nsplit = 1;
    while (nsplit > 1 && na_layout(units, nsplit, G).total > TD_NOALLOC_SCRATCH_BYTES)
        --nsplit;
    const int round = td::kTokPerRound;
    int chunk = ((top_k + nsplit - 1) / nsplit + round - 1) / round * round;
    nsplit = (top_k + chunk - 1) / chunk;
    const NaLayout L = na_layout(units, nsplit, G);
    if (chunk > td::kMaxSparseChunk || L.total > TD_NOALLOC_SCRATCH_BYTES)
        return TD_ERR_WORKSPACE_TOO_SMALL;  // beyond what the fixed scratch holds

    void *base = nullptr;
    td_status st = scratch_address(&base);
    if (st)
        return st;
    char *b = (char *)base;
    cudaStream_t cs = (cudaStream_t)stream;
    // tickets and status must start at zero; the array keeps the last call's contents
    if (cudaMemsetAsync(b, 0, L.part_m, cs) != cudaSuccess)
        return TD_ERR_CUDA;

    td::AttnArgs a{};
    a.q = (const uint16_t *)q;
    a.k = (const uint16_t *)k_cache;
    a.v = (const uint16_t *)v_cache;
    a.seq_lens = seq_lens;
    a.idx = idx;
    a.out = (uint16_t *)out;
    a.out_f32 = out_f32;
    a.scores = nullptr;
    a.part_m = (float *)(b + L.part_m);
    a.part_l = (float *)(b + L.part_l);
    a.part_o = (float *)(b + L.part_o);
    a.tickets = (uint32_t *)(b + L.tickets);
    a.status = (uint32_t *)(b + L.status);
    a.Hq = s.num_q_heads;
    a.Hkv = s.num_kv_heads;
    a.Nmax = s.max_seq_len;
    a.top_k = top_k;
    a.idx_dep = 1;
    a.chunk = chunk;
    a.nsplit = nsplit;
    a.scale = s.scale != 0.0f ? s.scale : 1.0f / sqrtf((float)s.head_dim);
    // the kernel td_sparse_attn takes by default: tensor cores for G = 4, 8
    const cudaError_t le =
        td::mma_supported(G) ? td::launch_attention_mma(G, true, false, kMmaSparseTokens, a, s.batch,
                                                        false, cs)
                             : td::launch_attention(G, true, false, false, false, a, s.batch,
                                                    false, cs);
    if (le != cudaSuccess)
        return TD_ERR_CUDA;
    return TD_OK;
}
