// spec_verify.cu -- libspecverify: batched draft-token verification by
// modified rejection sampling on one GB300 (sm_103a): host layer and C ABI.
//
// What it computes (the pages it follows):
//  * tech-tldr.com "投機的デコーディングとドラフトモデル", section
//    受理判定の数理：修正版棄却サンプリング -- keep x_i when r < min(1, p/q),
//    otherwise stop and draw from normalize(max(0, p - q));
//  * r-jc.jp "LLM推論の高速化｜KVキャッシュと投機的デコーディングを自作で実測",
//    section 投機的デコーディングとは -- p = probs(target row, T), ordered
//    tests, first-rejection break, residual (rejected) or bonus (all kept)
//    draw from row nacc; section 投機的デコーディングを実装して受理率と速度を実測
//    -- at T = 0 a proposal is kept iff it equals the target argmax;
//  * issoh.co.jp "Speculative Decoding（投機的デコーディング）とは？…", section
//    受理・棄却の規則と出力分布が変わらない理由, steps 1-5.
//
// One call = a 16-byte memset of the error word, the claim counter and the
// header-ready count on the stream + one kernel launch: the persistent cluster
// kernel (sv_sweep.cuh), or for V <= 1024 the warp-per-sequence kernel
// (sv_small.cuh).  The cluster kernel reads the rest of the per-call header
// (K, the claim order) from a pinned, device-mapped host buffer, copying it
// into the workspace first when the batch is larger than the grid; it draws
// the tokens and writes the outputs.  With sv_options.temperature_host, or
// for a batch of K = 0 sequences only (spec_sample), the host may launch its
// split variant, which walks sequences that read no draft rows on half
// clusters (run() says when).
#include <cuda_runtime.h>
#include <string.h>

#include <algorithm>
#include <map>
#include <mutex>
#include <tuple>
#include <vector>

#include "../../include/specverify.h"
#include "sv_small.cuh"
#include "sv_sweep.cuh"
#include "sv_tree.cuh"

namespace sv {

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
constexpr int kSmemPerCtaMax = 227 * 1024;   // opt-in dynamic shared memory limit
// A row (target and draft) must fit, resident, in the shared memory of one
// cluster of 16 CTAs: these limits leave room for the slices' rounding.
constexpr int kMaxVocabBf16 = 786432;
constexpr int kMaxVocabF32 = 393216;

struct Geom {
    int s = 0, nv = 0, ch = 0, nchunks = 0;
    int C = 0;          // CTAs per cluster (per row)
    int nw = 0;         // warps per CTA
    int kw = 0;         // chunks of the longest warp range
    int kc = 0;         // chunks of the longest CTA span
    int clusters = 0;   // persistent grid size (clusters)
    size_t smem = 0;
};

static int elem_size(sv_dtype dt) { return dt == SV_DTYPE_BF16 ? 2 : 4; }

// 16-byte vectors per lane per chunk (a chunk is 32 * nv * 16 bytes): 4 once
// V spans two such chunks, smaller for small vocabularies.
static int pick_nv(int V, int s)
{
    const int E = 16 / s;
    for (int nv = 4; nv > 1; nv >>= 1)
        if ((long long)V >= 2LL * 32 * nv * E)
            return nv;
    return 1;
}

static int chunk_elems(int V, int s) { return 32 * pick_nv(V, s) * (16 / s); }

static int n_chunks(int V, int s)
{
    const int ch = chunk_elems(V, s);
    return (V + ch - 1) / ch;
}

// ---- workspace layout: the per-call header (the first 16 bytes reset by
// every call; K, the order and the packed row starts written by the kernel
// from the mapped header, or uploaded from pageable staging) ----
struct WsLayout {
    size_t err, next_unit, ready, next_unit_g, K, order, seq_end, cu_t, cu_d, header_end, total;
};

static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

static bool ws_layout(int B, int Kmax, int V, sv_dtype dt, WsLayout* L)
{
    if (B < 0 || Kmax < 0 || Kmax > SV_K_MAX || V < 1)
        return false;
    (void)V;
    (void)dt;
    size_t o = 0;
    L->err = o;
    L->next_unit = o + 4;
    L->ready = o + 8;   // CTAs done copying the mapped header's K and order here
    L->next_unit_g = o + 12;   // the greedy queue's claim counter (split launches)
    o = align256(o + 16);
    L->K = o;        o = align256(o + (size_t)B * 4);
    L->order = o;    o = align256(o + (size_t)B * 4);
    L->seq_end = o;   // K and the order end here (the packed row starts follow)
    L->cu_t = o;     o = align256(o + (size_t)B * 4);
    L->cu_d = o;     o = align256(o + (size_t)B * 4);
    L->header_end = o;
    L->total = o;
    return true;
}

struct DeviceInfo {
    int nsm = 0;
    bool attrs_set[2][7] = {};
    void* static_scratch = nullptr;   // device address of g_static_scratch on this device
};

// Scratch of spec_verify_noalloc: a fixed device array in the library's own
// module (one copy per device, resolved once per device with
// cudaGetSymbolAddress), and the host array its per-call header is staged in.
// Neither needs initial contents: every call rewrites the header it uses.
static __device__ __align__(256) unsigned char g_static_scratch[SV_STATIC_SCRATCH_BYTES];
static unsigned char g_static_header[SV_STATIC_SCRATCH_BYTES];

static std::mutex g_mu;
static DeviceInfo g_dev[64];
// cudaOccupancyMaxActiveClusters per (device, kernel, cluster size, warps, smem)
static std::map<std::tuple<int, int, int, int, size_t>, int> g_fit;
// chosen geometry per (device, V, dtype, B, Kmax, tuning overrides)
static std::map<std::tuple<int, int, int, int, int, int, int, int, int>, Geom> g_pick;

template <typename T, int NV, bool WIDE, bool HOST, bool SPLIT = false>
static cudaError_t prepare_kernels(int dev)
{
    const int ti = sizeof(T) == 2 ? 1 : 0;
    const int ni = SPLIT ? 6 : NV == 1 ? 0 : NV == 2 ? 1 : (WIDE ? 3 : 2) + (HOST ? 2 : 0);
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_dev[dev].attrs_set[ti][ni]) {
        auto kern = sv_sweep_kernel<T, NV, WIDE, HOST, SPLIT>;
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             kSmemPerCtaMax);
        if (e != cudaSuccess)
            return e;
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess)
            return e;
        g_dev[dev].attrs_set[ti][ni] = true;
    }
    return cudaSuccess;
}

static void sweep_config(cudaLaunchConfig_t* cfg, cudaLaunchAttribute* attr, const Geom& g,
                         int clusters, cudaStream_t st)
{
    *cfg = cudaLaunchConfig_t{};
    cfg->gridDim = dim3((unsigned)(clusters * g.C), 1, 1);
    cfg->blockDim = dim3((unsigned)(32 * g.nw), 1, 1);
    cfg->dynamicSmemBytes = g.smem;
    cfg->stream = st;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)g.C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg->attrs = attr;
    cfg->numAttrs = 1;
}

// How many clusters of this shape the device holds at once (0: cannot launch).
template <typename T, int NV, bool WIDE, bool HOST>
static cudaError_t cluster_capacity(const Geom& g, int dev, int* n)
{
    cudaError_t e = prepare_kernels<T, NV, WIDE, HOST>(dev);
    if (e != cudaSuccess)
        return e;
    const auto key = std::make_tuple(dev, (int)sizeof(T) * 16 + NV + (HOST ? 256 : 0), g.C, g.nw, g.smem);
    {
        std::lock_guard<std::mutex> lk(g_mu);
        auto it = g_fit.find(key);
        if (it != g_fit.end()) {
            *n = it->second;
            return cudaSuccess;
        }
    }
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[1];
    sweep_config(&cfg, attr, g, 1, 0);
    int v = 0;
    e = cudaOccupancyMaxActiveClusters(&v, sv_sweep_kernel<T, NV, WIDE, HOST>, &cfg);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        v = 0;
    }
    std::lock_guard<std::mutex> lk(g_mu);
    g_fit[key] = v;
    *n = v;
    return cudaSuccess;
}

// host: the logits are device-mapped host memory (16-byte vectors only: the
// host path exists for NV = 4)
template <typename T>
static cudaError_t capacity_nv(const Geom& g, bool host, int dev, int* n)
{
    const bool wide = g.C * g.nw > 32;
    switch (g.nv) {
    case 1: return cluster_capacity<T, 1, false, false>(g, dev, n);
    case 2: return cluster_capacity<T, 2, false, false>(g, dev, n);
    default:
        if (host)
            return wide ? cluster_capacity<T, 4, true, true>(g, dev, n)
                        : cluster_capacity<T, 4, false, true>(g, dev, n);
        return wide ? cluster_capacity<T, 4, true, false>(g, dev, n)
                    : cluster_capacity<T, 4, false, false>(g, dev, n);
    }
}

// Geometry for C CTAs of nw warps per row: P = C * nw warp ranges of whole
// chunks (lengths differ by at most one); false if it does not fit.
static bool shape_geometry(int V, sv_dtype dt, int C, int nw, Geom* g)
{
    const int s = elem_size(dt);
    g->s = s;
    g->nv = pick_nv(V, s);
    g->ch = 32 * g->nv * (16 / s);
    g->nchunks = (V + g->ch - 1) / g->ch;
    if (C < 1 || C > kMaxCluster || nw < 1 || nw > kMaxWarps || C * nw > kMaxParts)
        return false;
    if (C > g->nchunks)   // no CTA without chunks
        return false;
    if (C * nw > 32 && g->nv != 4)   // more than 32 ranges: large vocabularies only
        return false;
    g->C = C;
    g->nw = nw;
    g->kw = (g->nchunks + C * nw - 1) / (C * nw);
    g->kc = cta_chunks(g->nchunks, C);
    const SweepLayout L = sweep_layout(nw, g->kc, g->kw, g->ch * s, C * nw);
    if (!sweep_layout_aligned(L))   // never launch a layout the kernel cannot address
        return false;
    g->smem = L.total;
    return g->smem <= (size_t)kSmemPerCtaMax;
}

static sv_status capacity_of(const Geom& g, sv_dtype dt, bool host, int dev, int* cap)
{
    const cudaError_t e = dt == SV_DTYPE_BF16 ? capacity_nv<__nv_bfloat16>(g, host, dev, cap)
                                              : capacity_nv<float>(g, host, dev, cap);
    return e == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

// Pick the geometry of one launch (cached per shape).  Every cluster size and
// warp count that fits is considered; a row's slice stays resident from its
// copy to its decision, so the device holds as many rows at once as clusters
// fit.  Score: rows in flight (resident clusters, up to B), then more warps
// per row (shorter passes), then larger clusters.  Tuning overrides: chunks
// per CTA (sets C), chunks per warp (sets the warps per CTA).
static sv_status pick_geometry(int V, sv_dtype dt, int B, int Kmax, int override_ncpc,
                               int want_cpw, int dev, bool host, Geom* g, int max_parts = kMaxParts)
{
    const auto key = std::make_tuple(dev, V, (int)dt, B, Kmax, override_ncpc, want_cpw, host ? 1 : 0, max_parts);
    {
        std::lock_guard<std::mutex> lk(g_mu);
        auto it = g_pick.find(key);
        if (it != g_pick.end()) {
            *g = it->second;
            return SV_OK;
        }
    }
    const int s = elem_size(dt);
    const int nch = n_chunks(V, s);
    Geom best;
    long long best_score = -1;
    for (int C = 1; C <= kMaxCluster; ++C) {
        if (override_ncpc > 0 && C != (nch + override_ncpc - 1) / override_ncpc)
            continue;
        for (int nw = 1; nw <= kMaxWarps && C * nw <= max_parts; ++nw) {
            if (want_cpw > 0) {
                const int ncpc = (nch + C - 1) / C;
                if (nw != std::min({(ncpc + want_cpw - 1) / want_cpw, kMaxParts / C, kMaxWarps}))
                    continue;
            }
            // without overrides, every warp range holds a chunk
            if (override_ncpc <= 0 && want_cpw <= 0 && C * nw > nch)
                continue;
            Geom t;
            if (!shape_geometry(V, dt, C, nw, &t))
                continue;
            int cap = 0;
            const sv_status st = capacity_of(t, dt, host, dev, &cap);
            if (st != SV_OK)
                return st;
            if (cap <= 0)
                continue;
            t.clusters = std::min(cap, std::max(1, B));
            const long long score = ((long long)t.clusters * 64 + C * nw) * 32 + C;
            if (score > best_score) {
                best_score = score;
                best = t;
            }
        }
    }
    (void)Kmax;
    if (best_score < 0)
        return SV_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_mu);
    g_pick[key] = best;
    *g = best;
    return SV_OK;
}

template <typename T, int NV, bool WIDE, bool HOST, bool SPLIT = false>
static cudaError_t launch_sweep(const Args& a, const Geom& g, cudaStream_t st, int dev)
{
    cudaError_t e = prepare_kernels<T, NV, WIDE, HOST, SPLIT>(dev);
    if (e != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[1];
    sweep_config(&cfg, attr, g, g.clusters, st);
    return cudaLaunchKernelEx(&cfg, sv_sweep_kernel<T, NV, WIDE, HOST, SPLIT>, a);
}

template <typename T>
static cudaError_t launch_nv(const Args& a, const Geom& g, bool host, cudaStream_t st, int dev)
{
    if (a.split_clusters > 0)   // (the host checked: NV = 4, at most 32 ranges, device rows)
        return launch_sweep<T, 4, false, false, true>(a, g, st, dev);
    const bool wide = g.C * g.nw > 32;
    switch (g.nv) {
    case 1: return launch_sweep<T, 1, false, false>(a, g, st, dev);
    case 2: return launch_sweep<T, 2, false, false>(a, g, st, dev);
    default:
        if (host)
            return wide ? launch_sweep<T, 4, true, true>(a, g, st, dev)
                        : launch_sweep<T, 4, false, true>(a, g, st, dev);
        return wide ? launch_sweep<T, 4, true, false>(a, g, st, dev)
                    : launch_sweep<T, 4, false, false>(a, g, st, dev);
    }
}

// Small vocabularies: one warp per sequence (sv_small.cuh), NE elements a
// lane (32 NE >= V).  The grid holds as many blocks of four warps as the
// device keeps resident (at most what the batch needs); a warp takes `tile`
// consecutive sequences at a time.
template <typename T, int NE>
static cudaError_t launch_small_ne(Args& a, int nsm, cudaStream_t st)
{
    static int occ[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return cudaErrorInvalidDevice;
    int per_sm;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        per_sm = occ[dev];
    }
    if (per_sm == 0) {
        cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, sv_small_kernel<T, NE>, 128, 0);
        if (e != cudaSuccess)
            return e;
        per_sm = std::max(per_sm, 1);
        std::lock_guard<std::mutex> lk(g_mu);
        occ[dev] = per_sm;
    }
    const long long max_warps = (long long)nsm * per_sm * 4;
    a.small_tile = (int)std::min<long long>(32, std::max<long long>(1, (a.B + max_warps - 1) / max_warps));
    const long long tiles = (a.B + a.small_tile - 1) / a.small_tile;
    const int blocks = (int)std::max<long long>(1, std::min<long long>((tiles + 3) / 4, (long long)nsm * per_sm));
    sv_small_kernel<T, NE><<<blocks, 128, 0, st>>>(a);
    return cudaGetLastError();
}

template <typename T>
static cudaError_t launch_small(Args& a, int nsm, cudaStream_t st)
{
    if (a.V <= 32)
        return launch_small_ne<T, 1>(a, nsm, st);
    if (a.V <= 64)
        return launch_small_ne<T, 2>(a, nsm, st);
    if (a.V <= 128)
        return launch_small_ne<T, 4>(a, nsm, st);
    if (a.V <= 256)
        return launch_small_ne<T, 8>(a, nsm, st);
    if (a.V <= 512)
        return launch_small_ne<T, 16>(a, nsm, st);
    return launch_small_ne<T, 32>(a, nsm, st);
}

static sv_status device_sms(int* dev_out, int* nsm_out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return SV_ERR_CUDA;
    int nsm;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        nsm = g_dev[dev].nsm;
    }
    if (nsm == 0) {
        if (cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return SV_ERR_CUDA;
        std::lock_guard<std::mutex> lk(g_mu);
        g_dev[dev].nsm = nsm;
    }
    *dev_out = dev;
    *nsm_out = nsm;
    return SV_OK;
}

// Device address of the static scratch on the current device (resolved on
// the first call per device).
static sv_status static_scratch(void** out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return SV_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_dev[dev].static_scratch) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || !p) {
            (void)cudaGetLastError();
            return SV_ERR_CUDA;
        }
        g_dev[dev].static_scratch = p;
    }
    *out = g_dev[dev].static_scratch;
    return SV_OK;
}

struct Call {
    const void* tgt;
    const void* drf;
    sv_dtype dtype;
    const int32_t* tok;
    const float* uni;
    const float* temp;
    int32_t B;
    const int32_t* K;
    int32_t V;
    int32_t* out_tok;
    int32_t* out_n;
};

static sv_status check_args(const Call& c, int* kmax_out)
{
    if (c.B < 0 || c.V < 1)
        return SV_ERR_INVALID_ARG;
    if (c.dtype != SV_DTYPE_F32 && c.dtype != SV_DTYPE_BF16)
        return SV_ERR_INVALID_ARG;
    if (c.B == 0) {
        *kmax_out = 0;
        return SV_OK;
    }
    if (!c.tgt || !c.uni || !c.temp || !c.K || !c.out_tok || !c.out_n)
        return SV_ERR_INVALID_ARG;
    int kmax = 0;
    for (int b = 0; b < c.B; ++b) {
        if (c.K[b] < 0 || c.K[b] > SV_K_MAX)
            return SV_ERR_INVALID_ARG;
        kmax = c.K[b] > kmax ? c.K[b] : kmax;
    }
    if (kmax > 0 && !c.tok)
        return SV_ERR_INVALID_ARG;
    if (c.V > sv_max_vocab(c.dtype))
        return SV_ERR_UNSUPPORTED;
    if ((long long)c.B * (kmax + 1) > (1LL << 30))
        return SV_ERR_UNSUPPORTED;
    *kmax_out = kmax;
    return SV_OK;
}

// Per host thread and device: pinned, device-mapped buffers the per-call
// header (K, the claim order, the packed row starts) is written to, used
// round-robin.  The kernel reads the header straight from the buffer (zero
// copy): a host-to-device copy on the copy engine, with the launch waiting on
// it, cost more than the few kilobytes warrant.  Only the 16 bytes of error
// word and claim counter are reset on the device, by a memset on the
// stream.  An event recorded after each launch guards a buffer's reuse, so a
// call blocks only if the GPU is kHeaderSlots calls behind.  The buffers live
// as long as the thread (they are small: the header is B * 16 bytes and up)
// and are released when it exits, once the kernels reading them are done.
constexpr int kHeaderSlots = 16;
struct HeaderSlot {
    unsigned char* buf = nullptr;
    unsigned char* dbuf = nullptr;   // its device address
    size_t cap = 0;
    cudaEvent_t done = nullptr;
    bool used = false;
};
struct HeaderRing {
    HeaderSlot slot[kHeaderSlots];
    int next = 0;
    ~HeaderRing()
    {
        for (HeaderSlot& s : slot) {
            if (s.used && s.done)
                (void)cudaEventSynchronize(s.done);   // a kernel may still read the buffer
            if (s.buf)
                (void)cudaFreeHost(s.buf);
            if (s.done)
                (void)cudaEventDestroy(s.done);
            s = HeaderSlot{};
        }
    }
};
static thread_local HeaderRing tl_header[64];

// A pinned slot of at least `need` bytes on device `dev` (nullptr if pinned
// memory is unavailable; the caller then stages in pageable memory).
static HeaderSlot* header_slot(int dev, size_t need, sv_status* st)
{
    HeaderRing& hr = tl_header[dev];
    *st = SV_OK;
    // a slot that is large enough and whose last kernel is done, nearest the
    // ring's position first: no allocation and no wait (each fresh slot of a
    // new size costs a page-locked allocation, milliseconds for a large batch)
    for (int k = 0; k < kHeaderSlots; ++k) {
        const int idx = (hr.next + k) % kHeaderSlots;
        HeaderSlot& s = hr.slot[idx];
        if (s.buf && s.cap >= need && s.done && (!s.used || cudaEventQuery(s.done) == cudaSuccess)) {
            s.used = false;
            hr.next = (idx + 1) % kHeaderSlots;
            return &s;
        }
    }
    (void)cudaGetLastError();   // a query that reported cudaErrorNotReady
    HeaderSlot& sl = hr.slot[hr.next];
    hr.next = (hr.next + 1) % kHeaderSlots;
    if (sl.used) {
        if (cudaEventSynchronize(sl.done) != cudaSuccess) {
            *st = SV_ERR_CUDA;
            return nullptr;
        }
        sl.used = false;
    }
    if (!sl.done && cudaEventCreateWithFlags(&sl.done, cudaEventDisableTiming) != cudaSuccess) {
        (void)cudaGetLastError();
        sl.done = nullptr;
        return nullptr;
    }
    if (sl.cap < need) {
        if (sl.buf)
            (void)cudaFreeHost(sl.buf);
        sl.buf = nullptr;
        sl.cap = 0;
        const size_t cap = std::max(need, (size_t)4096);
        if (cudaHostAlloc(reinterpret_cast<void**>(&sl.buf), cap, cudaHostAllocMapped) !=
            cudaSuccess) {
            (void)cudaGetLastError();
            sl.buf = nullptr;
            return nullptr;
        }
        if (cudaHostGetDevicePointer(reinterpret_cast<void**>(&sl.dbuf), sl.buf, 0) != cudaSuccess) {
            (void)cudaGetLastError();
            (void)cudaFreeHost(sl.buf);
            sl.buf = nullptr;
            sl.dbuf = nullptr;
            return nullptr;
        }
        sl.cap = cap;
    }
    return &sl;
}

// Headers of calls captured into CUDA graphs: a graph's kernel reads its
// header at every replay, so each capture takes a pinned slot of its own that
// is never written again (kept until the process ends).  Slots are allocated
// by ordinary calls (allocation is not allowed during a capture), so that a
// few of the size in use are always free.  The spare pool is bounded: when
// larger slots are added, the smallest spares beyond kCaptureSpareMax go
// (no kernel reads a spare slot).
struct CapturePool {
    std::vector<HeaderSlot*> free_slots;   // allocated, not yet taken by a capture
};
static CapturePool g_capture[64];
constexpr int kCaptureSpare = 4;
constexpr int kCaptureSpareMax = 8;

static void reserve_capture_slots(int dev, size_t need)
{
    std::lock_guard<std::mutex> lk(g_mu);
    auto& fs = g_capture[dev].free_slots;
    int fit = 0;
    for (HeaderSlot* h : fs)
        fit += h->cap >= need ? 1 : 0;
    if (fit >= kCaptureSpare)
        return;
    while ((int)fs.size() + (kCaptureSpare - fit) > kCaptureSpareMax) {
        size_t k_min = 0;   // the smallest spare that is too small for this shape
        bool found = false;
        for (size_t k = 0; k < fs.size(); ++k)
            if (fs[k]->cap < need && (!found || fs[k]->cap < fs[k_min]->cap)) {
                k_min = k;
                found = true;
            }
        if (!found)
            break;
        (void)cudaFreeHost(fs[k_min]->buf);
        delete fs[k_min];
        fs.erase(fs.begin() + (long)k_min);
    }
    for (; fit < kCaptureSpare; ++fit) {
        HeaderSlot* h = new HeaderSlot;
        const size_t cap = std::max(need, (size_t)4096);
        if (cudaHostAlloc(reinterpret_cast<void**>(&h->buf), cap, cudaHostAllocMapped) != cudaSuccess ||
            cudaHostGetDevicePointer(reinterpret_cast<void**>(&h->dbuf), h->buf, 0) != cudaSuccess) {
            (void)cudaGetLastError();
            if (h->buf)
                (void)cudaFreeHost(h->buf);
            delete h;
            return;
        }
        h->cap = cap;
        fs.push_back(h);
    }
}

// A slot for a call being captured (nullptr: none of this size was reserved).
static HeaderSlot* capture_slot(int dev, size_t need)
{
    std::lock_guard<std::mutex> lk(g_mu);
    auto& fs = g_capture[dev].free_slots;
    for (size_t k = 0; k < fs.size(); ++k) {
        if (fs[k]->cap >= need) {
            HeaderSlot* h = fs[k];
            fs.erase(fs.begin() + (long)k);
            return h;
        }
    }
    return nullptr;
}

// host_header: where the per-call header is assembled before its upload
// (nullptr: a pinned slot, else a pageable per-thread buffer).
// host_rows: the logits are device-mapped host memory (read in place).
static sv_status run(const Call& c, int kmax, const sv_options* opt, void* ws, size_t ws_bytes,
                     cudaStream_t stream, unsigned char* host_header = nullptr, bool host_rows = false)
{
    if (c.B == 0)
        return SV_OK;
    WsLayout L;
    if (!ws_layout(c.B, kmax, c.V, c.dtype, &L))
        return SV_ERR_INVALID_ARG;
    if (!ws || ws_bytes < L.total || ((uintptr_t)ws & 255))
        return SV_ERR_NO_MEMORY;
    int dev = 0, nsm = 0;
    sv_status st = device_sms(&dev, &nsm);
    if (st != SV_OK)
        return st;
    cudaStreamCaptureStatus cst = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cst) != cudaSuccess)
        return SV_ERR_CUDA;
    const bool capturing = cst != cudaStreamCaptureStatusNone;
    if (!host_rows && !capturing) {   // (not re-checked while a graph is captured)
        cudaPointerAttributes pa;
        if (cudaPointerGetAttributes(&pa, c.tgt) != cudaSuccess)
            return SV_ERR_CUDA;
        if (pa.type != cudaMemoryTypeDevice && pa.type != cudaMemoryTypeManaged)
            return SV_ERR_INVALID_ARG;
        if (pa.type == cudaMemoryTypeDevice && pa.device != dev)
            return SV_ERR_INVALID_ARG;
    }
    // small vocabularies: the warp-per-sequence kernel (no geometry, claims
    // or header copy); the tuning options, which shape the cluster sweep, and
    // the expired-wait test (it has no waits) do not apply to it
    const bool small = c.V <= kSmallVocab && !(opt && (opt->chunks_per_cta || opt->chunks_per_warp ||
                                                      opt->expire_copy_waits));
    Geom g;
    if (!small) {
        st = pick_geometry(c.V, c.dtype, c.B, kmax, opt ? opt->chunks_per_cta : 0,
                           opt ? opt->chunks_per_warp : 0, dev, host_rows, &g);
        if (st != SV_OK)
            return st;
        if (host_rows && g.nv != 4)   // the in-place path reads 16-byte vectors
            return SV_ERR_UNSUPPORTED;
        if ((long long)g.clusters * g.C > 0x7fffffffLL)
            return SV_ERR_UNSUPPORTED;
    }

    const sv_diag* dg = opt ? &opt->diag : nullptr;
    const bool want_diag = dg && (dg->p_x || dg->q_x || dg->resid_mass || dg->final_row);
    if (want_diag && ((dg->p_x == nullptr) != (dg->q_x == nullptr)))
        return SV_ERR_INVALID_ARG;   // p_x and q_x are written together

    // Header: zeroed error word and claim counter; K; the claim order
    // (sequences by K, longest first, so the tail holds short ones); the
    // packed row starts.
    thread_local std::vector<unsigned char> hdr_tls;
    unsigned char* hdr = host_header;
    HeaderSlot* slot = nullptr;
    if (capturing) {
        // a slot of the graph's own (reserved by an earlier ordinary call of
        // this size); pageable staging cannot be captured
        if (hdr)
            return SV_ERR_UNSUPPORTED;
        slot = capture_slot(dev, L.header_end);
        if (!slot)
            return SV_ERR_UNSUPPORTED;
        hdr = slot->buf;
    } else if (!hdr) {
        reserve_capture_slots(dev, L.header_end);
        sv_status hs = SV_OK;
        slot = header_slot(dev, L.header_end, &hs);
        if (hs != SV_OK)
            return hs;
        if (slot) {
            hdr = slot->buf;
        } else {
            hdr_tls.assign(L.header_end, 0);
            hdr = hdr_tls.data();
        }
    }
    const bool packed = opt && opt->packed_logits;
    const size_t up_bytes = packed ? L.header_end : L.seq_end;   // row starts only when packed
    memset(hdr, 0, L.K);   // error word, claim counter, ready count; every other field is written
    memcpy(hdr + L.K, c.K, (size_t)c.B * 4);
    // Split launch: given the caller's host copy of the temperatures, the
    // greedy sequences (T = 0) can go to split clusters, whose two halves
    // each walk greedy rows in the shared memory one sampling row takes.
    // Cg = clusters * nG / (nG + 6 nS) clusters are split: a sampling
    // sequence keeps a whole cluster about six times as long as a greedy one
    // keeps a half on the 1:1 mix of V = 128256 bf16 sequences, K ~ U{1..8};
    // the whole clusters take what is left of the greedy queue once the
    // sampling one is empty, so a low Cg costs less than a high one.  Only
    // plain calls split (no diagnostics, verify-all or tuning), and only when
    // the sampling sequences fill at least two waves of the whole clusters
    // (with fewer, the last long sampling sequences set the step's length: a
    // batch of 60 sampling and 196 greedy sequences took 59 us split against
    // 53 whole) and the greedy ones the halves' first wave.
    //
    // A batch of K = 0 sequences only (spec_sample: one bonus draw per row,
    // no draft rows) splits every cluster, with no hint needed, when it has
    // a sequence for each half's first wave.
    int split_cg = 0, split_ns = c.B;
    const float* th = opt ? opt->temperature_host : nullptr;
    const bool plain = !host_rows && !want_diag && !(opt && (opt->verify_all || opt->chunks_per_cta ||
                                                             opt->chunks_per_warp || opt->expire_copy_waits));
    const bool splittable = !small && plain && g.nv == 4 && g.nw % 2 == 0 && g.C * g.nw <= 32;
    bool all_k0 = kmax == 0;
    for (int b = 0; all_k0 && b < c.B; ++b)
        all_k0 = c.K[b] == 0;
    if (splittable && all_k0 && c.B >= 2 * g.clusters && 2 * g.clusters <= kFirstUnits) {
        split_cg = g.clusters;
        split_ns = 0;
    } else if (splittable && th && g.clusters >= 2) {
        int ng = 0;
        for (int b = 0; b < c.B; ++b)
            ng += th[b] == 0.0f ? 1 : 0;
        const int ns = c.B - ng;
        const long long cg = (long long)g.clusters * ng / ((long long)ng + 6LL * ns);
        const int cgi = (int)std::min<long long>({cg, (long long)g.clusters - 1, (long long)ng / 2});
        if (cgi >= 1 && ns >= 2 * (g.clusters - cgi) && g.clusters + cgi <= kFirstUnits) {
            split_cg = cgi;
            split_ns = ns;
        }
    }
    if (!small) {   // the claim order (the small-vocabulary kernel takes sequences in index order)
        // by K, longest first; split with a hint: the sampling sequences, then
        // the greedy ones
        int32_t* ord = reinterpret_cast<int32_t*>(hdr + L.order);
        int pos = 0;
        const bool by_kind = split_cg > 0 && split_ns > 0;   // (th is set: a hinted split)
        for (int cls = 0; cls < (by_kind ? 2 : 1); ++cls) {
            auto in = [&](int b) { return !by_kind || ((th[b] == 0.0f) == (cls == 1)); };
            int cnt[SV_K_MAX + 2] = {0};
            for (int b = 0; b < c.B; ++b)
                if (in(b))
                    ++cnt[SV_K_MAX - c.K[b] + 1];
            cnt[0] = pos;
            for (int k = 1; k <= SV_K_MAX + 1; ++k)
                cnt[k] += cnt[k - 1];
            for (int b = 0; b < c.B; ++b)
                if (in(b))
                    ord[cnt[SV_K_MAX - c.K[b]]++] = b;
            pos = cnt[SV_K_MAX + 1];   // this class's end: the next one's start
        }
    }
    if (packed) {
        int32_t* ct = reinterpret_cast<int32_t*>(hdr + L.cu_t);
        int32_t* cd = reinterpret_cast<int32_t*>(hdr + L.cu_d);
        long long rt = 0, rd = 0;
        for (int b = 0; b < c.B; ++b) {
            ct[b] = (int32_t)rt;
            cd[b] = (int32_t)rd;
            rt += c.K[b] + 1;
            rd += c.K[b];
        }
    }
    unsigned char* base = static_cast<unsigned char*>(ws);
    // where the kernel reads the header: the mapped slot itself (only the
    // error word and the claim counter live in the workspace), or the
    // workspace after an upload (pageable staging)
    const unsigned char* hbase = base;
    if (slot) {
        if (cudaMemsetAsync(base, 0, 16, stream) != cudaSuccess)
            return SV_ERR_CUDA;
        hbase = slot->dbuf;
    } else if (cudaMemcpyAsync(base, hdr, up_bytes, cudaMemcpyHostToDevice, stream) !=
               cudaSuccess) {
        return SV_ERR_CUDA;
    }

    Args a;
    a.tgt = c.tgt;
    a.drf = c.drf;
    a.tok = c.tok;
    a.uni = c.uni;
    a.temp = c.temp;
    a.out_tok = c.out_tok;
    a.out_n = c.out_n;
    a.B = c.B;
    a.Kmax = kmax;
    a.V = c.V;
    a.nchunks = g.nchunks;
    a.C = g.C;
    a.kw = g.kw;
    a.early_exit = (want_diag || (opt && opt->verify_all)) ? 0 : 1;
    a.has_draft = c.drf != nullptr ? 1 : 0;
    const uintptr_t al = (uintptr_t)c.tgt | (c.drf ? (uintptr_t)c.drf : 0);
    a.aligned = ((al & 15) == 0) && (((size_t)c.V * g.s) % 16 == 0);
    a.err = reinterpret_cast<uint32_t*>(base + L.err);
    a.next_unit = reinterpret_cast<int*>(base + L.next_unit);
    a.K = reinterpret_cast<const int32_t*>(hbase + L.K);
    a.order = reinterpret_cast<const int32_t*>(hbase + L.order);
    // the kernel copies K and the order from the mapped header into the
    // workspace (where the uploaded header already is for pageable staging),
    // when there are tickets to claim after the first wave: the claims then
    // read device memory instead of crossing the host link (with no claims
    // the copy only delayed the first rows: 2 us on a batch of one)
    a.copy_hdr = (!small && hbase != base && c.B > g.clusters) ? 1 : 0;
    a.ready = reinterpret_cast<int*>(base + L.ready);
    a.K_dev = reinterpret_cast<int32_t*>(base + L.K);
    a.order_dev = reinterpret_cast<int32_t*>(base + L.order);
    a.split_clusters = split_cg;
    a.split_ns = split_ns;
    a.next_unit_g = reinterpret_cast<int*>(base + L.next_unit_g);
    if (!small) {
        // first-wave slots: the first tickets of the queue (split: the
        // sampling queue's for the whole clusters, then the greedy queue's,
        // two for each split cluster)
        const int32_t* ord = reinterpret_cast<const int32_t*>(hdr + L.order);
        const int nfull = g.clusters - split_cg;
        const int nf = std::min(nfull, kFirstUnits);   // clusters <= B
        for (int k = 0; k < nf; ++k) {
            a.first_b[k] = ord[k];
            a.first_K[k] = c.K[ord[k]];
        }
        for (int k = 0; k < 2 * split_cg; ++k) {   // nfull + 2 split_cg <= kFirstUnits
            a.first_b[nfull + k] = ord[split_ns + k];
            a.first_K[nfull + k] = c.K[ord[split_ns + k]];
        }
    }
    a.p_x = want_diag ? dg->p_x : nullptr;
    a.q_x = want_diag ? dg->q_x : nullptr;
    a.resid = want_diag ? dg->resid_mass : nullptr;
    a.final_row = want_diag ? dg->final_row : nullptr;
    a.want_pq = a.p_x != nullptr ? 1 : 0;
    a.want_resid = a.resid != nullptr ? 1 : 0;
    a.want_final = a.final_row != nullptr ? 1 : 0;
    a.packed = packed ? 1 : 0;
    a.cu_t = reinterpret_cast<const int32_t*>(hbase + L.cu_t);
    a.cu_d = reinterpret_cast<const int32_t*>(hbase + L.cu_d);
    a.want_stats = (opt && opt->stats) ? 1 : 0;
    a.stats = a.want_stats ? reinterpret_cast<unsigned long long*>(opt->stats) : nullptr;
    a.want_kv = (opt && opt->kv_len) ? 1 : 0;
    a.expire_waits = (opt && opt->expire_copy_waits) ? 1 : 0;
    a.kv_len = a.want_kv ? opt->kv_len : nullptr;

    a.small_tile = 1;
    const cudaError_t e = small ? (c.dtype == SV_DTYPE_BF16 ? launch_small<__nv_bfloat16>(a, nsm, stream)
                                                            : launch_small<float>(a, nsm, stream))
                                : (c.dtype == SV_DTYPE_BF16 ? launch_nv<__nv_bfloat16>(a, g, host_rows, stream, dev)
                                                            : launch_nv<float>(a, g, host_rows, stream, dev));
    if (slot && !capturing) {   // the kernel reads the slot: it is free again once the kernel is done
        if (cudaEventRecord(slot->done, stream) != cudaSuccess)
            return SV_ERR_CUDA;
        slot->used = true;
    }
    return e == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

// The device's view of page-locked host memory mapped into its address space
// (nullptr for any other pointer).
static const void* mapped_host(const void* p)
{
    cudaPointerAttributes pa;
    if (cudaPointerGetAttributes(&pa, p) != cudaSuccess) {
        (void)cudaGetLastError();
        return nullptr;
    }
    return (pa.type == cudaMemoryTypeHost && pa.devicePointer) ? pa.devicePointer : nullptr;
}

// Launch geometry a call would use (for reports and tests).
static sv_status geometry_of(int B, int Kmax, int V, sv_dtype dt, int ncpc, int cpw,
                             int32_t* out)
{
    int dev = 0, nsm = 0;
    sv_status st = device_sms(&dev, &nsm);
    if (st != SV_OK)
        return st;
    Geom g;
    st = pick_geometry(V, dt, B, Kmax, ncpc, cpw, dev, false, &g);
    if (st != SV_OK)
        return st;
    out[0] = g.C;
    out[1] = g.nw;
    out[2] = g.kw;
    out[3] = g.clusters;
    out[4] = 32 * g.nw;
    out[5] = (int32_t)g.smem;
    out[6] = std::min(g.C * g.nw, g.nchunks);   // warp ranges holding chunks
    out[7] = g.nchunks;
    return SV_OK;
}

// ---------------------------------------------------------------------------
// token trees: one cluster per sequence (sv_tree_kernel)
// ---------------------------------------------------------------------------
template <typename T, int NV>
static cudaError_t launch_tree(const TreeArgs& ta, const Geom& g, size_t smem, cudaStream_t st)
{
    auto kern = sv_tree_kernel<T, NV>;
    static bool attrs_done[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return cudaErrorInvalidDevice;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if (!attrs_done[dev]) {
            cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 kSmemPerCtaMax);
            if (e != cudaSuccess)
                return e;
            e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
            if (e != cudaSuccess)
                return e;
            attrs_done[dev] = true;
        }
    }
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    // persistent: as many clusters as the device holds at once (at most B),
    // cluster c verifying sequence c, then claiming the next
    static std::map<std::tuple<int, int, int, size_t>, int> cap_cache;
    int cap = 0;
    {
        const auto key = std::make_tuple(dev, g.C, g.nw, smem);
        std::lock_guard<std::mutex> lk(g_mu);
        auto it = cap_cache.find(key);
        if (it != cap_cache.end()) {
            cap = it->second;
        } else {
            cudaLaunchConfig_t q = {};
            cudaLaunchAttribute qa[1];
            q.gridDim = dim3((unsigned)g.C, 1, 1);
            q.blockDim = dim3((unsigned)(32 * g.nw), 1, 1);
            q.dynamicSmemBytes = smem;
            qa[0].id = cudaLaunchAttributeClusterDimension;
            qa[0].val.clusterDim.x = (unsigned)g.C;
            qa[0].val.clusterDim.y = 1;
            qa[0].val.clusterDim.z = 1;
            q.attrs = qa;
            q.numAttrs = 1;
            if (cudaOccupancyMaxActiveClusters(&cap, kern, &q) != cudaSuccess) {
                (void)cudaGetLastError();
                cap = 0;
            }
            cap_cache[key] = cap;
        }
    }
    if (cap <= 0)
        return cudaErrorInvalidConfiguration;
    const int clusters = std::min(cap, ta.B);
    cfg.gridDim = dim3((unsigned)(clusters * g.C), 1, 1);
    cfg.blockDim = dim3((unsigned)(32 * g.nw), 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)g.C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, ta);
}

template <typename T>
static cudaError_t launch_tree_nv(const TreeArgs& ta, const Geom& g, size_t smem, cudaStream_t st)
{
    switch (g.nv) {
    case 1: return launch_tree<T, 1>(ta, g, smem, st);
    case 2: return launch_tree<T, 2>(ta, g, smem, st);
    default: return launch_tree<T, 4>(ta, g, smem, st);
    }
}

}  // namespace sv

// ---------------------------------------------------------------------------
// C ABI
// ---------------------------------------------------------------------------
extern "C" {

const char* sv_status_string(sv_status s)
{
    switch (s) {
    case SV_OK: return "SV_OK";
    case SV_ERR_INVALID_ARG: return "SV_ERR_INVALID_ARG";
    case SV_ERR_CUDA: return "SV_ERR_CUDA";
    case SV_ERR_UNSUPPORTED: return "SV_ERR_UNSUPPORTED";
    case SV_ERR_NO_MEMORY: return "SV_ERR_NO_MEMORY";
    case SV_ERR_TIMEOUT: return "SV_ERR_TIMEOUT";
    }
    return "SV_UNKNOWN_STATUS";
}

int32_t sv_abi_version(void) { return SV_ABI_VERSION; }

int32_t sv_max_vocab(sv_dtype dtype)
{
    if (dtype != SV_DTYPE_F32 && dtype != SV_DTYPE_BF16)
        return 0;
    return dtype == SV_DTYPE_BF16 ? sv::kMaxVocabBf16 : sv::kMaxVocabF32;
}

sv_status sv_geometry(int32_t B, int32_t Kmax, int32_t V, sv_dtype dtype, int32_t chunks_per_cta,
                      int32_t chunks_per_warp, int32_t* out8)
{
    if (!out8 || B < 1 || Kmax < 0 || Kmax > SV_K_MAX || V < 1 || chunks_per_cta < 0 ||
        chunks_per_warp < 0 ||
        (dtype != SV_DTYPE_F32 && dtype != SV_DTYPE_BF16))
        return SV_ERR_INVALID_ARG;
    if (V > sv_max_vocab(dtype))
        return SV_ERR_UNSUPPORTED;
    return sv::geometry_of(B, Kmax, V, dtype, chunks_per_cta, chunks_per_warp, out8);
}

size_t sv_workspace_size(int32_t B, int32_t Kmax, int32_t V, sv_dtype dtype)
{
    if (dtype != SV_DTYPE_F32 && dtype != SV_DTYPE_BF16)
        return 0;
    sv::WsLayout L;
    if (!sv::ws_layout(B, Kmax, V, dtype, &L))
        return 0;
    return L.total;
}

sv_status spec_verify_ex(const void* target_logits, const void* draft_logits, sv_dtype dtype,
                         const int32_t* draft_tokens, const float* uniforms,
                         const float* temperature, int32_t B, const int32_t* K, int32_t V,
                         int32_t* out_tokens, int32_t* out_num_accepted,
                         const sv_options* options, void* workspace, size_t workspace_bytes,
                         cudaStream_t stream)
{
    const sv::Call c{target_logits, draft_logits, dtype, draft_tokens, uniforms, temperature,
                     B, K, V, out_tokens, out_num_accepted};
    int kmax = 0;
    const sv_status st = sv::check_args(c, &kmax);
    if (st != SV_OK)
        return st;
    if (options && (options->chunks_per_cta < 0 || options->chunks_per_warp < 0))
        return SV_ERR_INVALID_ARG;
    if (options && ((((uintptr_t)options->stats) & 7) || (((uintptr_t)options->kv_len) & 3)))
        return SV_ERR_INVALID_ARG;   // 64-bit counters, 32-bit lengths
    if (options && (options->packed_logits < 0 || options->packed_logits > 1))
        return SV_ERR_INVALID_ARG;
    if (options && (options->expire_copy_waits < 0 || options->expire_copy_waits > 1))
        return SV_ERR_INVALID_ARG;
    if (options && options->packed_logits) {
        long long rows = 0;   // row indices of the packed arrays must fit 32 bits
        for (int b = 0; b < B; ++b)
            rows += (long long)K[b] + 1;
        if (rows > 0x7fffffffLL)
            return SV_ERR_UNSUPPORTED;
    }
    return sv::run(c, kmax, options, workspace, workspace_bytes, stream);
}

size_t sv_sample_workspace_size(int32_t B, int32_t V, sv_dtype dtype)
{
    const size_t ws = sv_workspace_size(B, 0, V, dtype);
    if (!ws)
        return 0;
    return ws + sv::align256((size_t)(B > 0 ? B : 1) * 4);   // + the per-row validity words
}

sv_status spec_sample(const void* logits, sv_dtype dtype, const float* uniforms,
                      const float* temperature, int32_t B, int32_t V, int32_t* out_tokens,
                      void* workspace, size_t workspace_bytes, cudaStream_t stream)
{
    if (B < 0)
        return SV_ERR_INVALID_ARG;
    // a K = 0 verification of every row: row 0 is the final draw, from p
    thread_local std::vector<int32_t> zeros;
    zeros.assign((size_t)B, 0);
    const size_t ws_bytes = sv_workspace_size(B, 0, V, dtype);
    int32_t* out_n = (workspace && ws_bytes) ? reinterpret_cast<int32_t*>(
                                                   static_cast<unsigned char*>(workspace) + ws_bytes)
                                             : nullptr;
    const sv::Call c{logits, nullptr, dtype, nullptr, uniforms, temperature,
                     B, zeros.data(), V, out_tokens, out_n ? out_n : out_tokens};
    int kmax = 0;
    const sv_status st = sv::check_args(c, &kmax);
    if (st != SV_OK || B == 0)
        return st;
    const size_t need = sv_sample_workspace_size(B, V, dtype);
    if (!workspace || !need || workspace_bytes < need || ((uintptr_t)workspace & 255))
        return SV_ERR_NO_MEMORY;
    return sv::run(c, 0, nullptr, workspace, ws_bytes, stream);
}

sv_status spec_verify_ws(const void* target_logits, const void* draft_logits, sv_dtype dtype,
                         const int32_t* draft_tokens, const float* uniforms,
                         const float* temperature, int32_t B, const int32_t* K, int32_t V,
                         int32_t* out_tokens, int32_t* out_num_accepted, void* workspace,
                         size_t workspace_bytes, cudaStream_t stream)
{
    return spec_verify_ex(target_logits, draft_logits, dtype, draft_tokens, uniforms, temperature,
                          B, K, V, out_tokens, out_num_accepted, nullptr, workspace,
                          workspace_bytes, stream);
}

sv_status spec_verify(const void* target_logits, const void* draft_logits, sv_dtype dtype,
                      const int32_t* draft_tokens, const float* uniforms, const float* temperature,
                      int32_t B, const int32_t* K, int32_t V, int32_t* out_tokens,
                      int32_t* out_num_accepted, cudaStream_t stream)
{
    const sv::Call c{target_logits, draft_logits, dtype, draft_tokens, uniforms, temperature,
                     B, K, V, out_tokens, out_num_accepted};
    int kmax = 0;
    sv_status st = sv::check_args(c, &kmax);
    if (st != SV_OK || B == 0)
        return st;
    const size_t bytes = sv_workspace_size(B, kmax, V, dtype);
    void* ws = nullptr;
    if (cudaMallocAsync(&ws, bytes, stream) != cudaSuccess) {
        (void)cudaGetLastError();
        return SV_ERR_NO_MEMORY;
    }
    st = sv::run(c, kmax, nullptr, ws, bytes, stream);
    if (cudaFreeAsync(ws, stream) != cudaSuccess && st == SV_OK)
        st = SV_ERR_CUDA;
    return st;
}

sv_status spec_verify_noalloc(const void* target_logits, const void* draft_logits, sv_dtype dtype,
                              const int32_t* draft_tokens, const float* uniforms,
                              const float* temperature, int32_t B, const int32_t* K, int32_t V,
                              int32_t* out_tokens, int32_t* out_num_accepted, cudaStream_t stream)
{
    const sv::Call c{target_logits, draft_logits, dtype, draft_tokens, uniforms, temperature,
                     B, K, V, out_tokens, out_num_accepted};
    int kmax = 0;
    sv_status st = sv::check_args(c, &kmax);
    if (st != SV_OK || B == 0)
        return st;
    const size_t bytes = sv_workspace_size(B, kmax, V, dtype);
    if (bytes == 0)
        return SV_ERR_INVALID_ARG;
    if (bytes > SV_STATIC_SCRATCH_BYTES)
        return SV_ERR_NO_MEMORY;   // this shape needs more scratch than the static array holds
    void* ws = nullptr;
    st = sv::static_scratch(&ws);
    if (st != SV_OK)
        return st;
    return sv::run(c, kmax, nullptr, ws, SV_STATIC_SCRATCH_BYTES, stream, sv::g_static_header);
}

sv_status sv_workspace_errors(void* workspace, uint32_t* flags, cudaStream_t stream)
{
    if (!workspace || !flags)
        return SV_ERR_INVALID_ARG;
    uint32_t v = 0;
    if (cudaMemcpyAsync(&v, workspace, 4, cudaMemcpyDeviceToHost, stream) != cudaSuccess)
        return SV_ERR_CUDA;
    if (cudaStreamSynchronize(stream) != cudaSuccess)
        return SV_ERR_CUDA;
    if (cudaMemsetAsync(workspace, 0, 4, stream) != cudaSuccess)
        return SV_ERR_CUDA;
    *flags = v;
    return (v & sv::kErrWaitTimeout) ? SV_ERR_TIMEOUT : (v & sv::kErrHint) ? SV_ERR_INVALID_ARG : SV_OK;
}

size_t sv_host_staging_size(int32_t B, int32_t Kmax, int32_t V, sv_dtype dtype)
{
    const size_t ws = sv_workspace_size(B, Kmax, V, dtype);
    if (!ws)
        return 0;
    const size_t s = (size_t)sv::elem_size(dtype);
    const size_t Bz = (size_t)B, K1 = (size_t)Kmax + 1, Vz = (size_t)V;
    return sv::align256(Bz * K1 * Vz * s) + sv::align256(Bz * (K1 - 1) * Vz * s) +
           sv::align256(Bz * (K1 - 1) * 4) + sv::align256(Bz * K1 * 4) + sv::align256(Bz * 4) +
           sv::align256(Bz * K1 * 4) + sv::align256(Bz * 4) + ws;
}

sv_status spec_verify_host(const void* h_target_logits, const void* h_draft_logits,
                           sv_dtype dtype, const int32_t* h_draft_tokens, const float* h_uniforms,
                           const float* h_temperature, int32_t B, const int32_t* K, int32_t V,
                           int32_t* h_out_tokens, int32_t* h_out_num_accepted,
                           void* device_staging, size_t staging_bytes, cudaStream_t stream)
{
    const sv::Call hc{h_target_logits, h_draft_logits, dtype, h_draft_tokens, h_uniforms,
                      h_temperature, B, K, V, h_out_tokens, h_out_num_accepted};
    int kmax = 0;
    sv_status st = sv::check_args(hc, &kmax);
    if (st != SV_OK || B == 0)
        return st;
    const size_t need = sv_host_staging_size(B, kmax, V, dtype);
    if (!device_staging || staging_bytes < need || ((uintptr_t)device_staging & 255))
        return SV_ERR_NO_MEMORY;
    cudaStreamCaptureStatus cst = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cst) != cudaSuccess)
        return SV_ERR_CUDA;
    if (cst != cudaStreamCaptureStatusNone)   // the call synchronises: not capturable
        return SV_ERR_UNSUPPORTED;
    const size_t s = (size_t)sv::elem_size(dtype);
    const size_t Bz = (size_t)B, K1 = (size_t)kmax + 1, Vz = (size_t)V;
    unsigned char* p = static_cast<unsigned char*>(device_staging);
    const size_t n_tgt = Bz * K1 * Vz * s, n_drf = Bz * (K1 - 1) * Vz * s;
    const size_t n_tok = Bz * (K1 - 1) * 4, n_uni = Bz * K1 * 4, n_tmp = Bz * 4;
    const size_t n_otok = Bz * K1 * 4, n_on = Bz * 4;
    unsigned char* d_tgt = p;                   p += sv::align256(n_tgt);
    unsigned char* d_drf = p;                   p += sv::align256(n_drf);
    unsigned char* d_tok = p;                   p += sv::align256(n_tok);
    unsigned char* d_uni = p;                   p += sv::align256(n_uni);
    unsigned char* d_tmp = p;                   p += sv::align256(n_tmp);
    unsigned char* d_otok = p;                  p += sv::align256(n_otok);
    unsigned char* d_on = p;                    p += sv::align256(n_on);
    void* ws = p;
    const size_t ws_bytes = staging_bytes - (size_t)(p - static_cast<unsigned char*>(device_staging));
    const bool has_drf = h_draft_logits && n_drf;
    // page-locked logits mapped into the device's address space are read in
    // place by the kernel, only the rows the method reaches; others are
    // copied into the staging first
    const void* m_tgt = sv::mapped_host(h_target_logits);
    const void* m_drf = has_drf ? sv::mapped_host(h_draft_logits) : nullptr;
    const bool in_place = m_tgt && (!has_drf || m_drf) && sv::pick_nv(V, (int)s) == 4;
    if ((!in_place &&
         (cudaMemcpyAsync(d_tgt, h_target_logits, n_tgt, cudaMemcpyHostToDevice, stream) != cudaSuccess ||
          (has_drf && cudaMemcpyAsync(d_drf, h_draft_logits, n_drf, cudaMemcpyHostToDevice, stream) !=
                          cudaSuccess))) ||
        (n_tok && cudaMemcpyAsync(d_tok, h_draft_tokens, n_tok, cudaMemcpyHostToDevice, stream) != cudaSuccess) ||
        cudaMemcpyAsync(d_uni, h_uniforms, n_uni, cudaMemcpyHostToDevice, stream) != cudaSuccess ||
        cudaMemcpyAsync(d_tmp, h_temperature, n_tmp, cudaMemcpyHostToDevice, stream) != cudaSuccess)
        return SV_ERR_CUDA;
    const void* tgt = in_place ? m_tgt : d_tgt;
    const void* drf = has_drf ? (in_place ? m_drf : d_drf) : nullptr;
    const sv::Call dc{tgt, drf, dtype,
                      n_tok ? reinterpret_cast<const int32_t*>(d_tok) : nullptr,
                      reinterpret_cast<const float*>(d_uni), reinterpret_cast<const float*>(d_tmp),
                      B, K, V, reinterpret_cast<int32_t*>(d_otok), reinterpret_cast<int32_t*>(d_on)};
    st = sv::run(dc, kmax, nullptr, ws, ws_bytes, stream, nullptr, in_place);
    if (st != SV_OK)
        return st;
    if (cudaMemcpyAsync(h_out_tokens, d_otok, n_otok, cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
        cudaMemcpyAsync(h_out_num_accepted, d_on, n_on, cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
        cudaStreamSynchronize(stream) != cudaSuccess)
        return SV_ERR_CUDA;
    return SV_OK;
}

size_t sv_tree_workspace_size(void) { return 256; }

sv_status spec_verify_tree(const void* target_logits, const void* draft_logits, sv_dtype dtype,
                           const int32_t* tokens, const int32_t* parent, const float* uniforms,
                           const float* temperature, int32_t B, int32_t Nmax, const int32_t* n_nodes,
                           int32_t V, int32_t* out_tokens, int32_t* out_path, int32_t* out_len,
                           void* workspace, size_t workspace_bytes, cudaStream_t stream)
{
    if (B < 0 || V < 1 || Nmax < 1 || Nmax > sv::kTreeMaxNodes ||
        (dtype != SV_DTYPE_F32 && dtype != SV_DTYPE_BF16))
        return SV_ERR_INVALID_ARG;
    if (B == 0)
        return SV_OK;
    if (!target_logits || !tokens || !parent || !uniforms || !temperature || !n_nodes || !out_tokens ||
        !out_path || !out_len)
        return SV_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < sv_tree_workspace_size() || ((uintptr_t)workspace & 255))
        return SV_ERR_NO_MEMORY;
    if (V > sv_max_vocab(dtype) || (long long)B * Nmax > (1LL << 30) || (long long)B * 16 > 0x7fffffffLL)
        return SV_ERR_UNSUPPORTED;
    int dev = 0, nsm = 0;
    sv_status st = sv::device_sms(&dev, &nsm);
    if (st != SV_OK)
        return st;
    sv::Geom g;
    // at most 32 warp ranges a row: one partial per lane in the combines
    st = sv::pick_geometry(V, dtype, 1 << 20, 0, 0, 0, dev, false, &g, 32);
    if (st != SV_OK)
        return st;
    const sv::SweepLayout L = sv::sweep_layout(g.nw, g.kc, g.kw, g.ch * g.s, g.C * g.nw);
    const size_t smem = sv::tree_smem_bytes(L, g.nw);
    if (smem > (size_t)sv::kSmemPerCtaMax)
        return SV_ERR_UNSUPPORTED;
    if (cudaMemsetAsync(workspace, 0, 16, stream) != cudaSuccess)
        return SV_ERR_CUDA;
    sv::TreeArgs ta;
    ta.tgt = target_logits;
    ta.drf = draft_logits;
    ta.tok = tokens;
    ta.parent = parent;
    ta.uni = uniforms;
    ta.temp = temperature;
    ta.n_nodes = n_nodes;
    ta.out_tok = out_tokens;
    ta.out_path = out_path;
    ta.out_len = out_len;
    ta.err = static_cast<uint32_t*>(workspace);
    ta.next = reinterpret_cast<int*>(static_cast<unsigned char*>(workspace) + 4);
    ta.B = B;
    ta.Nmax = Nmax;
    ta.V = V;
    ta.nchunks = g.nchunks;
    ta.C = g.C;
    ta.kw = g.kw;
    const uintptr_t al = (uintptr_t)target_logits | (draft_logits ? (uintptr_t)draft_logits : 0);
    ta.aligned = ((al & 15) == 0) && (((size_t)V * g.s) % 16 == 0);
    ta.has_draft = draft_logits != nullptr ? 1 : 0;
    const cudaError_t e = dtype == SV_DTYPE_BF16 ? sv::launch_tree_nv<__nv_bfloat16>(ta, g, smem, stream)
                                                 : sv::launch_tree_nv<float>(ta, g, smem, stream);
    return e == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

}  // extern "C"
