// sv_sweep.cuh -- the persistent verification kernel.
//
// A grid of thread-block clusters (C CTAs of nw warps each, as many as the
// device holds at once) works through the batch one row (sequence b, position
// i) at a time per cluster.  The row's vocabulary is cut into P = C * nw
// contiguous ranges of whole chunks whose lengths differ by at most one; warp
// g = rank * nw + w owns range g and keeps its slice of the row (target and
// draft) resident in its own part of the CTA's shared memory, filled by one
// 1-D bulk copy (cp.async.bulk) per array that completes on the warp's
// mbarrier.  No two warps share data, so the steady state has no CTA-wide
// barrier at all.
//
// Schedule: a cluster walks one sequence's positions in order.  Row i+1 is
// read only once x_i has been accepted (the method's own early exit: rows after
// the first rejection are never read).  Cluster c starts with ticket c (its
// sequence and K in the launch arguments); later sequences come from one
// atomic claim each (longest K first), made by rank 0 a row ahead and handed
// to the cluster with that row's exchange while two waves of tickets remain,
// else when the current sequence ends (so the last go to the clusters free
// first).  A split launch (the caller's host copy of the temperatures) turns
// the last clusters into two half-walkers each, which take the greedy
// sequences from a queue of their own, two greedy rows in the shared memory
// one sampling row takes; a batch of K = 0 sequences only splits every
// cluster (see the SPLIT flag of the kernel).
//
// Per row, each warp makes one pass over its slice, from shared memory
// straight into registers (the chunk loops are not unrolled: the smaller loop
// body ran workload 4 3% and workload 2 7% faster):
//   greedy row       lane max (packed bf16x2 / three-input fp32 max), the
//                    first chunk holding it, then the lowest index holding it;
//   tested sampling  sums of the target and draft weights exp2(fma(l, c, -r))
//   row              (c = log2(e)/T) weighed against the proposal's own logits
//                    (r = l_x c), so no maximum is needed and every warp's
//                    partials add; a row whose weights overflow is weighed
//                    again against its maxima; packed two-lane fp32;
//   bonus row        the warp's maximum, then per-strip sums of the target's
//                    weights against it, kept for the draw.
// exchange  every warp pushes a 16-byte partial to every CTA of the cluster
//           with st.async, completing on the receiver's exchange mbarrier
//           (double-buffered by row parity);
// decide    every warp combines all P partials (identical arithmetic, so
//           identical results) and decides u q(x) < p(x), or x == argmax at
//           temperature 0;
// residual  rejected rows (every tested row in verify-all mode): per-strip
//           sums of max(0, p - q) and the warp's sum of p, from the resident
//           slice, and a second exchange of the per-warp totals;
// draw      at the sequence's final row the warp whose range holds u * S (a
//           compensated prefix over the warps, then over its strips in index
//           order, then over the lanes of one strip, then inside the lane)
//           picks the token by inverse CDF from its resident slice and writes
//           the sequence's outputs.
#pragma once

#include "sv_common.cuh"

namespace sv {

constexpr int kMaxParts = 64;   // warps per row: lanes j and j + 32 hold partials j, j + 32 in the combines

// Warp range g of a row of `nchunks` chunks cut into P ranges is chunks
// [range_lo(g), range_lo(g + 1)): lengths floor or ceil of nchunks / P.  The
// nw ranges of CTA r are contiguous and span at most cta_chunks() chunks.
__host__ __device__ inline int range_lo(int g, int nchunks, int P)
{
    return (int)(((long long)g * nchunks) / P);
}

__host__ __device__ inline int cta_chunks(int nchunks, int C) { return (nchunks + C - 1) / C; }

// Dynamic shared memory of one CTA (host and device compute it alike).
struct SweepLayout {
    size_t region_bytes;   // the CTA's span of target chunks (kc of them); the draft
                           // chunks follow in a second region of the same size
    size_t bars;           // [nw] slot mbarriers
    size_t xbar;           // [2] exchange mbarriers: row partials
    size_t xbar2;          // [2] exchange mbarriers: residual totals
    size_t xbarc;          // mbarrier of a claim made between sequences
    size_t xbuf;           // [2][P] float4 row partials (P = warps per row)
    size_t xbuf2;          // [2][P] float2 residual totals
    size_t xclaim;         // [2] int2: (sequence, ticket) claimed by rank 0 during the row
    size_t first;          // int2: (sequence, ticket) of a claim made between sequences
    size_t stats;          // [nw][kw][strips][4] float: per-strip partial sums of the
                           // draw masses (at most 64 bytes a chunk; kw = longest range)
    size_t total;
};

__host__ __device__ inline SweepLayout sweep_layout(int nw, int kc, int kw, int chunk_bytes, int P)
{
    SweepLayout L;
    L.region_bytes = (size_t)kc * (size_t)chunk_bytes;
    size_t o = 2 * L.region_bytes;
    L.bars = o;
    o += (size_t)nw * 8;
    L.xbar = o;
    o += 16;
    L.xbar2 = o;
    o += 16;
    L.xbarc = o;
    o += 8;
    o = (o + 15) & ~(size_t)15;
    L.xbuf = o;
    o += 2 * (size_t)P * 16;
    L.xbuf2 = o;
    o += 2 * (size_t)P * 8;
    L.xclaim = o;
    o += 16;
    L.first = o;
    o += 8;
    o = (o + 15) & ~(size_t)15;   // stats are read as 16-byte vectors
    L.stats = o;
    o += (size_t)nw * kw * 8 * 8;
    L.total = o;
    return L;
}

// The alignments the kernel's shared-memory accesses rely on: 16-byte
// vectors (slices, row partials, strip partials), 8-byte mbarriers, residual
// totals and claims.  Chunks are whole multiples of 16 bytes, so every
// warp's slice starts 16-byte aligned inside its region.
__host__ __device__ inline bool sweep_layout_aligned(const SweepLayout& L)
{
    return L.region_bytes % 16 == 0 && L.bars % 8 == 0 && L.xbar % 8 == 0 && L.xbar2 % 8 == 0 &&
           L.xbarc % 8 == 0 && L.xbuf % 16 == 0 && L.xbuf2 % 8 == 0 && L.xclaim % 8 == 0 &&
           L.first % 8 == 0 &&
           L.stats % 16 == 0;
}

// Row flags, from the sequence's K_b and T alone.
enum : int {
    kFGreedy = 1,   // T == 0
    kFTest = 2,     // i < K_b: a proposal is tested at this row
    kFDraft = 4,    // the draft row is read (tested sampling row)
    kFUsable = 8,   // temperature usable and, if needed, draft logits supplied
    kFMaxRef = 16   // tested row weighed against the row maxima (its weights
                    // against the proposal's logits overflowed)
};

struct Row {
    int i, b, Kb;
    float T;
    int flags;
    int tb, db;   // rows of position 0 of sequence b in the target / draft arrays
};

__device__ __forceinline__ Row make_row(const Args& a, int i, int b, int Kb, float T, int tb, int db)
{
    Row r;
    r.i = i;
    r.b = b;
    r.Kb = Kb;
    r.T = T;
    r.tb = tb;
    r.db = db;
    const int greedy = T == 0.0f ? kFGreedy : 0;
    const int test = i < Kb ? kFTest : 0;
    const int draft = (test && !greedy) ? kFDraft : 0;
    const int usable = (temperature_usable(T) && (!draft || a.has_draft != 0)) ? kFUsable : 0;
    r.flags = greedy | test | draft | usable;
    return r;
}

// A sequence's draft tokens and uniforms, lane j holding position j
// (K_max <= 32), loaded once per sequence when it is claimed, so that no row
// waits on them.
struct SeqVals {
    int tok;
    float u;
};

__device__ __forceinline__ SeqVals seq_vals(const Args& a, int b, int lane)
{
    SeqVals v{0, 0.0f};
    if (lane < a.Kmax)
        v.tok = __ldg(a.tok + (size_t)b * a.Kmax + lane);
    if (lane <= a.Kmax)
        v.u = __ldg(a.uni + (size_t)b * (a.Kmax + 1) + lane);
    return v;
}

// The row's proposal, held by lane 0 of every warp: token and uniform (from
// the sequence's registers) and the bits of the two logits at the token
// (loaded when the row's copies are issued, widened to fp32 where first used,
// after the slice has arrived).
struct Tok {
    int x;
    float u;
    uint32_t lt, ld;
    int ok;
};

// Whole warp (shuffles); the result is meaningful in every lane.
__device__ __forceinline__ Tok tok_of(const Args& a, const Row& r, const SeqVals& sv)
{
    const int x = __shfl_sync(kFull, sv.tok, r.i & 31);
    const float u = __shfl_sync(kFull, sv.u, r.i & 31);
    Tok t{0, 0.0f, 0u, 0u, 0};
    if (!(r.flags & kFUsable))
        return t;
    if (!(r.flags & kFTest)) {
        t.ok = 1;
        return t;
    }
    t.x = x;
    bool ok = x >= 0 && x < a.V;
    if (!(r.flags & kFGreedy)) {
        t.u = u;
        ok = ok && u >= 0.0f && u < 1.0f;
    }
    t.ok = ok ? 1 : 0;
    return t;
}

// The logits at the proposed token: a tested sampling row's pass weighs its
// logits against them, and its decision needs them.  Greedy rows need
// neither (loading them anyway made their pass wait for the load).
template <typename T>
__device__ __forceinline__ void tok_logits(const Args& a, const Row& r, Tok& t)
{
    if (!t.ok || !(r.flags & kFTest) || (r.flags & kFGreedy))
        return;
    const size_t trow = (size_t)r.tb + r.i;
    t.lt = Elem<T>::load_raw(static_cast<const T*>(a.tgt) + trow * (size_t)a.V + t.x);
    if (r.flags & kFDraft)
        t.ld = Elem<T>::load_raw(static_cast<const T*>(a.drf) +
                                 ((size_t)r.db + r.i) * (size_t)a.V + t.x);
}

// The proposal as every lane sees it, the logits widened to fp32.
struct TokF {
    int x;
    float u, lt, ld;
    int ok;
};

template <typename T>
__device__ __forceinline__ TokF shfl_tok(const Tok& t)
{
    TokF o;
    o.x = __shfl_sync(kFull, t.x, 0);
    o.u = __shfl_sync(kFull, t.u, 0);
    o.lt = Elem<T>::widen(__shfl_sync(kFull, t.lt, 0));
    o.ld = Elem<T>::widen(__shfl_sync(kFull, t.ld, 0));
    o.ok = __shfl_sync(kFull, t.ok, 0);
    return o;
}

// The per-call header's K and claim order: the device copies once every CTA
// has written its slice (`ok`, sticky per thread, set by one acquire load),
// else the pinned, device-mapped header itself (a round trip over the host
// link).  Both hold the same values, so either read is correct.
__device__ __forceinline__ bool header_on_device(const Args& a, bool& ok)
{
    if (!ok && a.copy_hdr) {
        int v;
        asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(a.ready) : "memory");
        ok = v >= (int)gridDim.x;
    }
    return ok;
}

__device__ __forceinline__ int header_order(const Args& a, int t, bool& ok)
{
    return header_on_device(a, ok) ? __ldcg(a.order_dev + t) : __ldg(a.order + t);
}

__device__ __forceinline__ int header_K(const Args& a, int b, bool& ok)
{
    return header_on_device(a, ok) ? __ldcg(a.K_dev + b) : __ldg(a.K + b);
}

// Claims (one thread): a ticket now, its sequence later (the ticket's value
// is not waited for until the sequence is needed).  The first wave's tickets
// 0 .. n_clusters - 1 are the clusters' own; the counter hands out the rest.
// Tickets past the batch, or anything out of range, read as -1.
__device__ __forceinline__ int claim_ticket(const Args& a, int n_clusters)
{
    return atomicAdd(a.next_unit, 1) + n_clusters;
}

__device__ __forceinline__ int ticket_unit(const Args& a, int t, bool& ok)
{
    if (t < 0 || t >= a.B)
        return -1;
    const int b = header_order(a, t, ok);
    return (b >= 0 && b < a.B) ? b : -1;
}

// The same in two steps, so that the order lookup's latency hides behind
// other work: the load (at a clamped index, always in bounds; B >= 1), then
// the range checks once its value is needed.
__device__ __forceinline__ int ticket_load(const Args& a, int t, bool& ok)
{
    return header_order(a, min(max(t, 0), a.B - 1), ok);
}

__device__ __forceinline__ int ticket_check(const Args& a, int t, int b)
{
    return (t >= 0 && t < a.B && b >= 0 && b < a.B) ? b : -1;
}

// A sequence's first row: K_b and T loaded at claim time, used when it starts.
struct UnitPos {
    int b, Kb;
    float T;
    int tb, db;
};

// The rows of position 0 of sequence b: computed for the padded layout,
// loaded for the packed one.
__device__ __forceinline__ int seq_trow(const Args& a, int b)
{
    return a.packed ? __ldg(a.cu_t + b) : b * (a.Kmax + 1);
}

__device__ __forceinline__ int seq_drow(const Args& a, int b)
{
    return a.packed ? __ldg(a.cu_d + b) : b * a.Kmax;
}

__device__ __forceinline__ UnitPos unit_pos(const Args& a, int b, bool& ok)
{
    return UnitPos{b, header_K(a, b, ok), __ldg(a.temp + b), seq_trow(a, b), seq_drow(a, b)};
}

// The first sequence of cluster `cid` (ticket cid): from the launch
// arguments for the first kFirstUnits clusters, else from the header.
__device__ __forceinline__ UnitPos first_unit_pos(const Args& a, int cid, int b, bool& ok)
{
    if (cid < kFirstUnits)
        return UnitPos{b, a.first_K[cid], __ldg(a.temp + b), seq_trow(a, b), seq_drow(a, b)};
    return unit_pos(a, b, ok);
}

// A half of a split cluster takes only sequences that read no draft rows
// (greedy ones, and K = 0 ones: a bonus draw alone), since its slices have no
// draft region: a sequence in its queue that has draft rows to read (the
// caller's temperature hint called it greedy, but its device temperature is
// not 0) is made unusable (outputs -1) and flagged in the error word.
__device__ __forceinline__ Row no_draft_only(const Args& a, Row r, int lane)
{
    if (r.flags & kFDraft) {
        r.flags &= ~kFUsable;
        if (lane == 0)
            atomicOr(a.err, kErrHint);
    }
    return r;
}

// The sequence's final-draw uniform (slot K_b), sampling sequences only.
__device__ __forceinline__ float final_uniform(const Args& a, const Row& r)
{
    if ((r.flags & kFGreedy) || !(r.flags & kFUsable))
        return 0.0f;
    return __ldg(a.uni + (size_t)r.b * (a.Kmax + 1) + r.Kb);
}

// ---------------------------------------------------------------------------
// per-lane chunk arithmetic on registers.  A lane holds NV 16-byte vectors of
// a chunk: elements (k * 32 + lane) * E .. + E - 1 for vector k.
// ---------------------------------------------------------------------------
template <typename T, int NV> struct Lane;

template <int NV> struct Lane<__nv_bfloat16, NV> {
    static constexpr int E = 8;
    // NaN-propagating max of the lane's 8 * NV elements
    __device__ static __forceinline__ float max(const uint4 (&v)[NV])
    {
        uint32_t m0 = bmax2_nan(v[0].x, v[0].y), m1 = bmax2_nan(v[0].z, v[0].w);
#pragma unroll
        for (int k = 1; k < NV; ++k) {
            m0 = bmax2_nan(m0, bmax2_nan(v[k].x, v[k].y));
            m1 = bmax2_nan(m1, bmax2_nan(v[k].z, v[k].w));
        }
        const uint32_t m = bmax2_nan(m0, m1);
        return max_nan(__uint_as_float(m << 16), __uint_as_float(m & 0xffff0000u));
    }
    // the two elements of a bf16 pair as fp32 (lower index in the low lane)
    __device__ static __forceinline__ uint64_t pair(uint32_t w)
    {
        return f2_pack(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
    }
    // sum of weight(l, m, c) over the lane's elements
    __device__ static __forceinline__ float exp_sum(const uint4 (&v)[NV], float m, float c)
    {
        const float r = ref_of(m, c);
        const uint64_t Cc = f2_pack(c, c), NR = f2_pack(-r, -r);
        uint64_t acc0 = f2_pack(0.0f, 0.0f), acc1 = acc0;
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const uint32_t wv[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                float d0, d1;
                f2_unpack(f2_fma(pair(wv[h]), Cc, NR), d0, d1);
                const uint64_t e = f2_pack(ex2_approx(d0), ex2_approx(d1));
                if (h & 1)
                    acc1 = f2_add(acc1, e);
                else
                    acc0 = f2_add(acc0, e);
            }
        }
        float a0, a1, b0, b1;
        f2_unpack(acc0, a0, a1);
        f2_unpack(acc1, b0, b1);
        return (a0 + a1) + (b0 + b1);
    }
    // element j (0 .. 8 * NV - 1, in index order) of the lane's slice
    __device__ static __forceinline__ float elem(const uint4 (&v)[NV], int j)
    {
        const uint4 q = v[j >> 3];
        const int h = (j >> 1) & 3;
        const uint32_t wd = h == 0 ? q.x : h == 1 ? q.y : h == 2 ? q.z : q.w;
        return (j & 1) ? __uint_as_float(wd & 0xffff0000u) : __uint_as_float(wd << 16);
    }
    // per strip (vector k: 8 elements), the lane's sum of weight(l, m, c)
    __device__ static __forceinline__ void exp_strips(const uint4 (&v)[NV], float m, float c, float (&s)[NV])
    {
        const float r = ref_of(m, c);
        const uint64_t Cc = f2_pack(c, c), NR = f2_pack(-r, -r);
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const uint32_t wv[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
            uint64_t acc0 = f2_pack(0.0f, 0.0f), acc1 = acc0;
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                float d0, d1;
                f2_unpack(f2_fma(pair(wv[h]), Cc, NR), d0, d1);
                const uint64_t e = f2_pack(ex2_approx(d0), ex2_approx(d1));
                if (h & 1)
                    acc1 = f2_add(acc1, e);
                else
                    acc0 = f2_add(acc0, e);
            }
            float a0, a1, b0, b1;
            f2_unpack(acc0, a0, a1);
            f2_unpack(acc1, b0, b1);
            s[k] = (a0 + a1) + (b0 + b1);
        }
    }
    // the residual term max(0, p - q) and the weight of p of element e of a
    // lane vector pair; the target and draft weights share a packed fma and
    // a packed multiply (the one rounding sequence of every residual term)
    __device__ static __forceinline__ void resid_term2(uint32_t wt, uint32_t wd, int half, uint64_t Cc,
                                                       uint64_t NR, uint64_t IS, float& r, float& et)
    {
        const float lt = half ? __uint_as_float(wt & 0xffff0000u) : __uint_as_float(wt << 16);
        const float ld = half ? __uint_as_float(wd & 0xffff0000u) : __uint_as_float(wd << 16);
        float a0, a1;
        f2_unpack(f2_fma(f2_pack(lt, ld), Cc, NR), a0, a1);
        et = ex2_approx(a0);
        float p, q;
        f2_unpack(f2_mul(f2_pack(et, ex2_approx(a1)), IS), p, q);
        r = fmaxf(__fsub_rn(p, q), 0.0f);
    }
    // per strip, the lane's sum of residual terms; over all strips, the
    // lane's sum of the weights of p.  Element pairs of each word: the same
    // per-element steps as resid_term2 (fma, ex2, multiply by the inverse
    // sum, subtract, clamp), fewer instructions.
    __device__ static __forceinline__ void resid_strips(const uint4 (&t)[NV], const uint4 (&d)[NV],
                                                        float mt, float ist, float md, float isd,
                                                        float c, float (&rs)[NV], float& ps)
    {
        const uint64_t Cc = f2_pack(c, c);
        const float rt = ref_of(mt, c), rd = ref_of(md, c);
        const uint64_t NT = f2_pack(-rt, -rt), ND = f2_pack(-rd, -rd);
        const uint64_t IT = f2_pack(ist, ist), ID = f2_pack(isd, isd);
        uint64_t pacc = f2_pack(0.0f, 0.0f);
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const uint32_t wt[4] = {t[k].x, t[k].y, t[k].z, t[k].w};
            const uint32_t wd[4] = {d[k].x, d[k].y, d[k].z, d[k].w};
            uint64_t racc = f2_pack(0.0f, 0.0f);
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                float a0, a1, b0, b1;
                f2_unpack(f2_fma(pair(wt[h]), Cc, NT), a0, a1);
                f2_unpack(f2_fma(pair(wd[h]), Cc, ND), b0, b1);
                const uint64_t et = f2_pack(ex2_approx(a0), ex2_approx(a1));
                const uint64_t ed = f2_pack(ex2_approx(b0), ex2_approx(b1));
                float r0, r1;
                f2_unpack(f2_sub(f2_mul(et, IT), f2_mul(ed, ID)), r0, r1);
                racc = f2_add(racc, f2_pack(fmaxf(r0, 0.0f), fmaxf(r1, 0.0f)));
                pacc = f2_add(pacc, et);
            }
            float r0, r1;
            f2_unpack(racc, r0, r1);
            rs[k] = r0 + r1;
        }
        float p0, p1;
        f2_unpack(pacc, p0, p1);
        ps = p0 + p1;
    }
    __device__ static __forceinline__ void resid_elem(const uint4& t, const uint4& d, int e, uint64_t Cc,
                                                      uint64_t NR, uint64_t IS, float& r, float& et)
    {
        const int h = e >> 1;
        const uint32_t wt = h == 0 ? t.x : h == 1 ? t.y : h == 2 ? t.z : t.w;
        const uint32_t wd = h == 0 ? d.x : h == 1 ? d.y : h == 2 ? d.z : d.w;
        resid_term2(wt, wd, e & 1, Cc, NR, IS, r, et);
    }
    // element e (0..7) of a lane vector, as fp32
    __device__ static __forceinline__ float vec_elem(const uint4& q, int e)
    {
        const int h = e >> 1;
        const uint32_t wd = h == 0 ? q.x : h == 1 ? q.y : h == 2 ? q.z : q.w;
        return (e & 1) ? __uint_as_float(wd & 0xffff0000u) : __uint_as_float(wd << 16);
    }
};

template <int NV> struct Lane<float, NV> {
    static constexpr int E = 4;
    __device__ static __forceinline__ float max(const uint4 (&v)[NV])
    {
        float m = max_nan(__uint_as_float(v[0].x), __uint_as_float(v[0].y));
        m = max3_nan(m, __uint_as_float(v[0].z), __uint_as_float(v[0].w));
#pragma unroll
        for (int k = 1; k < NV; ++k) {
            m = max3_nan(m, __uint_as_float(v[k].x), __uint_as_float(v[k].y));
            m = max3_nan(m, __uint_as_float(v[k].z), __uint_as_float(v[k].w));
        }
        return m;
    }
    __device__ static __forceinline__ float exp_sum(const uint4 (&v)[NV], float m, float c)
    {
        const float r = ref_of(m, c);
        const uint64_t Cc = f2_pack(c, c), NR = f2_pack(-r, -r);
        uint64_t acc0 = f2_pack(0.0f, 0.0f), acc1 = acc0;
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            float d0, d1, d2, d3;
            f2_unpack(f2_fma(f2_pack(__uint_as_float(v[k].x), __uint_as_float(v[k].y)), Cc, NR), d0, d1);
            f2_unpack(f2_fma(f2_pack(__uint_as_float(v[k].z), __uint_as_float(v[k].w)), Cc, NR), d2, d3);
            acc0 = f2_add(acc0, f2_pack(ex2_approx(d0), ex2_approx(d1)));
            acc1 = f2_add(acc1, f2_pack(ex2_approx(d2), ex2_approx(d3)));
        }
        float a0, a1, b0, b1;
        f2_unpack(acc0, a0, a1);
        f2_unpack(acc1, b0, b1);
        return (a0 + a1) + (b0 + b1);
    }
    __device__ static __forceinline__ float elem(const uint4 (&v)[NV], int j)
    {
        const uint4 q = v[j >> 2];
        const int h = j & 3;
        return __uint_as_float(h == 0 ? q.x : h == 1 ? q.y : h == 2 ? q.z : q.w);
    }
    __device__ static __forceinline__ void exp_strips(const uint4 (&v)[NV], float m, float c, float (&s)[NV])
    {
        const float r = ref_of(m, c);
        const uint64_t Cc = f2_pack(c, c), NR = f2_pack(-r, -r);
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            float d0, d1, d2, d3;
            f2_unpack(f2_fma(f2_pack(__uint_as_float(v[k].x), __uint_as_float(v[k].y)), Cc, NR), d0, d1);
            f2_unpack(f2_fma(f2_pack(__uint_as_float(v[k].z), __uint_as_float(v[k].w)), Cc, NR), d2, d3);
            float a0, a1, b0, b1;
            f2_unpack(f2_pack(ex2_approx(d0), ex2_approx(d1)), a0, a1);
            f2_unpack(f2_pack(ex2_approx(d2), ex2_approx(d3)), b0, b1);
            s[k] = (a0 + a1) + (b0 + b1);
        }
    }
    __device__ static __forceinline__ void resid_term2(uint32_t wt, uint32_t wd, int /*half*/, uint64_t Cc,
                                                       uint64_t NR, uint64_t IS, float& r, float& et)
    {
        float a0, a1;
        f2_unpack(f2_fma(f2_pack(__uint_as_float(wt), __uint_as_float(wd)), Cc, NR), a0, a1);
        et = ex2_approx(a0);
        float p, q;
        f2_unpack(f2_mul(f2_pack(et, ex2_approx(a1)), IS), p, q);
        r = fmaxf(__fsub_rn(p, q), 0.0f);
    }
    __device__ static __forceinline__ void resid_strips(const uint4 (&t)[NV], const uint4 (&d)[NV],
                                                        float mt, float ist, float md, float isd,
                                                        float c, float (&rs)[NV], float& ps)
    {
        const uint64_t Cc = f2_pack(c, c);
        const float rt = ref_of(mt, c), rd = ref_of(md, c);
        const uint64_t NT = f2_pack(-rt, -rt), ND = f2_pack(-rd, -rd);
        const uint64_t IT = f2_pack(ist, ist), ID = f2_pack(isd, isd);
        uint64_t pacc = f2_pack(0.0f, 0.0f);
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const uint64_t tp[2] = {f2_pack(__uint_as_float(t[k].x), __uint_as_float(t[k].y)),
                                    f2_pack(__uint_as_float(t[k].z), __uint_as_float(t[k].w))};
            const uint64_t dp[2] = {f2_pack(__uint_as_float(d[k].x), __uint_as_float(d[k].y)),
                                    f2_pack(__uint_as_float(d[k].z), __uint_as_float(d[k].w))};
            uint64_t racc = f2_pack(0.0f, 0.0f);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                float a0, a1, b0, b1;
                f2_unpack(f2_fma(tp[h], Cc, NT), a0, a1);
                f2_unpack(f2_fma(dp[h], Cc, ND), b0, b1);
                const uint64_t et = f2_pack(ex2_approx(a0), ex2_approx(a1));
                const uint64_t ed = f2_pack(ex2_approx(b0), ex2_approx(b1));
                float r0, r1;
                f2_unpack(f2_sub(f2_mul(et, IT), f2_mul(ed, ID)), r0, r1);
                racc = f2_add(racc, f2_pack(fmaxf(r0, 0.0f), fmaxf(r1, 0.0f)));
                pacc = f2_add(pacc, et);
            }
            float r0, r1;
            f2_unpack(racc, r0, r1);
            rs[k] = r0 + r1;
        }
        float p0, p1;
        f2_unpack(pacc, p0, p1);
        ps = p0 + p1;
    }
    __device__ static __forceinline__ void resid_elem(const uint4& t, const uint4& d, int e, uint64_t Cc,
                                                      uint64_t NR, uint64_t IS, float& r, float& et)
    {
        const uint32_t wt = e == 0 ? t.x : e == 1 ? t.y : e == 2 ? t.z : t.w;
        const uint32_t wd = e == 0 ? d.x : e == 1 ? d.y : e == 2 ? d.z : d.w;
        resid_term2(wt, wd, 0, Cc, NR, IS, r, et);
    }
    __device__ static __forceinline__ float vec_elem(const uint4& q, int e)
    {
        return __uint_as_float(e == 0 ? q.x : e == 1 ? q.y : e == 2 ? q.z : q.w);
    }
};

template <typename T, int NV>
__device__ __forceinline__ void load_chunk(const T* p, int lane, uint4 (&v)[NV])
{
    const uint4* q = reinterpret_cast<const uint4*>(p);
#pragma unroll
    for (int k = 0; k < NV; ++k)
        v[k] = q[k * 32 + lane];
}

// Per-strip partial sums of a chunk for the draw: v[k] is the lane's sum
// over strip k (vector k of every lane).  Three butterfly levels, halving the
// values each lane carries while there is more than one (a transpose-reduce:
// four shuffles for four strips), leave each strip's sum as four partials
// (partial q over the eight lanes whose lane index is q modulo 4), stored as
// dst[k * 4 + q].  SINGLE: two more levels add the four partials, and the
// strip's sum is stored alone as dst[k] (a quarter of the space).
template <int NV, bool SINGLE = false>
__device__ __forceinline__ void strip_partials(const float (&v)[NV], int lane, float* dst)
{
    float x;
    int k;
    if constexpr (NV == 4) {
        const bool b4 = (lane & 16) != 0, b3 = (lane & 8) != 0;
        // xor 16: the lower half keeps strips 0, 1, the upper half 2, 3
        const float r0 = __shfl_xor_sync(kFull, b4 ? v[0] : v[2], 16);
        const float r1 = __shfl_xor_sync(kFull, b4 ? v[1] : v[3], 16);
        const float k0 = (b4 ? v[2] : v[0]) + r0, k1 = (b4 ? v[3] : v[1]) + r1;
        // xor 8: each lane keeps one strip, 2 * b4 + b3
        const float r2 = __shfl_xor_sync(kFull, b3 ? k0 : k1, 8);
        x = (b3 ? k1 : k0) + r2;
        k = (b4 ? 2 : 0) + (b3 ? 1 : 0);
    } else if constexpr (NV == 2) {
        const bool b4 = (lane & 16) != 0;
        x = (b4 ? v[1] : v[0]) + __shfl_xor_sync(kFull, b4 ? v[0] : v[1], 16);
        x += __shfl_xor_sync(kFull, x, 8);
        k = b4 ? 1 : 0;
    } else {
        x = v[0] + __shfl_xor_sync(kFull, v[0], 16);
        x += __shfl_xor_sync(kFull, x, 8);
        k = 0;
    }
    x += __shfl_xor_sync(kFull, x, 4);
    const int keep = NV == 4 ? 4 : (NV == 2 ? 12 : 28);   // lanes holding a distinct partial
    if constexpr (SINGLE) {
        x += __shfl_xor_sync(kFull, x, 1);
        x += __shfl_xor_sync(kFull, x, 2);
        if ((lane & (keep | 3)) == 0)
            dst[k] = x;
    } else {
        if ((lane & keep) == 0)
            dst[k * 4 + (lane & 3)] = x;
    }
}

// Warp sum of non-negative lane sums, compensated; +inf if a lane overflowed
// (and no lane is NaN), NaN if a lane is NaN.
__device__ __forceinline__ float sum_or_special(float v)
{
    if (__any_sync(kFull, isnan(v)))
        return NAN;
    if (__any_sync(kFull, isinf(v)))
        return INFINITY;
    return warp_sum_comp(v);
}

// sum_or_special of two values, interleaved (each result as the single form).
__device__ __forceinline__ void sum_or_special2(float& va, float& vb)
{
    const bool nan_a = __any_sync(kFull, isnan(va)), nan_b = __any_sync(kFull, isnan(vb));
    const bool inf_a = __any_sync(kFull, isinf(va)), inf_b = __any_sync(kFull, isinf(vb));
    warp_sum_comp2(va, vb);
    va = nan_a ? NAN : (inf_a ? INFINITY : va);
    vb = nan_b ? NAN : (inf_b ? INFINITY : vb);
}

// Merge part (m2, s2) into (m, s): the larger maximum, both sums taken
// against it (a part at -inf holds no mass).
__device__ __forceinline__ void merge_ms(float& m, float& s, float m2, float s2, float c)
{
    const float M = max_nan(m, m2);
    const float a = m == -INFINITY ? 0.0f : (m == M ? s : s * weight(m, M, c));
    const float b = m2 == -INFINITY ? 0.0f : (m2 == M ? s2 : s2 * weight(m2, M, c));
    m = M;
    s = a + b;
}

// Combine two sets of (max, sum relative to that max) parts held one per
// lane, interleaved so that their shuffle latencies overlap; the sums are
// compensated.  Every lane gets the same results.
__device__ __forceinline__ void combine_ms2(float ma_part, float sa_part, float mb_part, float sb_part,
                                            float c, float& ma, float& Sa, float& mb, float& Sb)
{
    ma = ma_part;
    mb = mb_part;
    warp_max_nan2(ma, mb);
    Sa = ma_part == -INFINITY ? 0.0f : (ma_part == ma ? sa_part : sa_part * weight(ma_part, ma, c));
    Sb = mb_part == -INFINITY ? 0.0f : (mb_part == mb ? sb_part : sb_part * weight(mb_part, mb, c));
    warp_sum_comp2(Sa, Sb);
}

// Inverse-CDF selection over `n` non-negative masses D(0..n-1), one warp:
// the smallest j with t < D(0) + ... + D(j), sums compensated, 32 at a time.
// `t` is reduced to the mass left inside the selected entry.  If t lies beyond
// the total (rounding), the last positive entry is taken and *beyond is set.
// Returns -1 if no entry is positive.  Every lane gets the same result.
template <typename F>
__device__ __forceinline__ int select_cdf(int n, F D, float& t, bool& beyond, int lane)
{
    int last_pos = -1;
    if (!beyond) {
        float base_s = 0.0f, base_c = 0.0f;   // compensated mass of earlier groups
        for (int j0 = 0; j0 < n; j0 += 32) {
            const int j = j0 + lane;
            const float d = j < n ? D(j) : 0.0f;
            if (d > 0.0f)
                last_pos = j;
            float s, c;
            warp_incl_scan_comp(d, lane, s, c);
            const float rel = (t - base_s) - base_c;   // mass left after earlier groups
            // an entry without mass is never taken (a remainder that rounded
            // below zero lands on the first entry with mass)
            const unsigned hit = __ballot_sync(kFull, j < n && d > 0.0f && rel < s + c);
            if (hit) {
                const int src = __ffs(hit) - 1;
                const float ex_s = __shfl_sync(kFull, s, src), ex_c = __shfl_sync(kFull, c, src);
                const float dd = __shfl_sync(kFull, d, src);
                t = rel - ((ex_s - dd) + ex_c);   // mass left inside the entry
                return j0 + src;
            }
            const float gs = __shfl_sync(kFull, s, 31), gc = __shfl_sync(kFull, c, 31);
            float ts, te;
            two_sum(base_s, gs, ts, te);
            base_s = ts;
            base_c += gc + te;
        }
    } else {
        for (int j0 = 0; j0 < n; j0 += 32) {
            const int j = j0 + lane;
            if (j < n && D(j) > 0.0f)
                last_pos = j;
        }
    }
    beyond = true;
    return __reduce_max_sync(kFull, last_pos);
}

// The element of one strip of a chunk that holds the point tc of the
// distribution drawn from (one warp; tv / dv: each lane's vector of the strip
// in the target / draft slice, dv read only for the residual).  The strip's
// index order is lane, then element, so: each lane's E terms, a compensated
// warp scan of their sums, the lane that holds the point, then its element.
// The terms are computed exactly as in the residual pass (or the bonus pass).
// Returns lane * E + e, or -1 if the strip has no mass; when the point lies
// beyond the strip's mass (rounding, or `beyond` already set) the last
// element with mass is taken.  NEAR: also set `near` (every lane): the point
// lies within `band` of a bound of the element taken (always so beyond the
// mass); without NEAR the distances are not tracked.
template <typename T, int NV, bool NEAR>
__device__ __forceinline__ int pick_in_strip(const uint4& tv, const uint4& dv, bool use_r, float m_t,
                                             float inv_st, float m_d, float inv_sd, float c, float tc,
                                             bool beyond, int lane, float band, bool& near)
{
    using LN = Lane<T, NV>;
    constexpr int E = Elem<T>::E;
    const float rt = ref_of(m_t, c), rd = ref_of(m_d, c);
    const uint64_t Cc = f2_pack(c, c), NR = f2_pack(-rt, -rd), IS = f2_pack(inv_st, inv_sd);
    float tm[E];
    float ls = 0.0f;
    int lastpos = -1;
#pragma unroll
    for (int e = 0; e < E; ++e) {
        float v;
        if (use_r) {
            float et;
            LN::resid_elem(tv, dv, e, Cc, NR, IS, v, et);
        } else {
            v = ex2_approx(__fmaf_rn(LN::vec_elem(tv, e), c, -rt));
        }
        tm[e] = v;
        ls += v;
        if (v > 0.0f)
            lastpos = lane * E + e;
    }
    int cand = -1;
    if (!beyond) {
        float ss, sc;
        warp_incl_scan_comp(ls, lane, ss, sc);
        const unsigned hit = __ballot_sync(kFull, ls > 0.0f && tc < ss + sc);
        if (hit) {
            const int src = __ffs(hit) - 1;
            const float tl = tc - ((ss - ls) + sc);   // the point's place in the lane (src)
            int ce = -1, lp = -1;
            float cum = 0.0f, dlo = 0.0f, dhi = 0.0f;   // the point's distances to ce's bounds
#pragma unroll
            for (int e = 0; e < E; ++e) {   // the same sums as ls
                const float prev = cum;
                cum += tm[e];
                if (tm[e] > 0.0f) {
                    lp = e;
                    if (ce < 0 && tl < cum) {
                        ce = e;
                        if (NEAR) {
                            dlo = tl - prev;
                            dhi = cum - tl;
                        }
                    }
                }
            }
            if (ce < 0) {   // rounding: the lane's last element with mass, at its bound
                ce = lp;
                dlo = 0.0f;
            }
            cand = __shfl_sync(kFull, lane * E + ce, src);
            if (NEAR)
                near = __shfl_sync(kFull, fminf(dlo, dhi) < band ? 1 : 0, src) != 0;
        }
    }
    if (cand < 0) {   // beyond the mass (rounding): the strip's last element with mass
        cand = __reduce_max_sync(kFull, lastpos);
        near = true;
    }
    return cand;
}

// Whether the draw's point lies within `band` of a bound of the token the
// pick takes (the same pick, with the distances tracked): a separate call,
// made only when counters are requested, so the draw path itself is the
// plain pick.
template <typename T, int NV>
__device__ __noinline__ bool draw_is_near(uint4 tv, uint4 dv, bool use_r, float m_t, float inv_st, float m_d,
                                          float inv_sd, float c, float tc, bool beyond, int lane, float band)
{
    bool near = false;
    (void)pick_in_strip<T, NV, true>(tv, dv, use_r, m_t, inv_st, m_d, inv_sd, c, tc, beyond, lane, band, near);
    return near;
}

// WIDE: more than 32 warp ranges per row (lanes hold two partials each in
// the combines); the host launches it for exactly those geometries.  HOST:
// the logits are device-mapped host memory, read with 16-byte loads instead
// of bulk copies (and never prefetched into L2).  SPLIT: the last
// a.split_clusters clusters of the grid are split in two halves (warps
// 0 .. nw/2 - 1 and nw/2 .. nw - 1 of every CTA), each half an independent
// row walker over half the warp ranges, its slices in one region (target or
// draft) of the CTA: they take the greedy sequences, which read no draft
// rows, from a queue of their own (order entries from a.split_ns on; the
// sampling sequences come first), two greedy rows in the shared memory one
// row of a sampling sequence takes.  The other clusters take the sampling
// queue, then what is left of the greedy one.  A batch of K = 0 sequences
// only (bonus draws, no draft rows) is split whole: a.split_clusters is the
// grid, a.split_ns is 0, and the halves keep one sum per strip for the draw.
template <typename T, int NV, bool WIDE, bool HOST, bool SPLIT = false>
__global__ void __maxnreg__(kMaxRegs) sv_sweep_kernel(const Args a)
{
    using EL = Elem<T>;
    using LN = Lane<T, NV>;
    constexpr int E = EL::E;
    constexpr int CH = 32 * NV * E;
    extern __shared__ __align__(128) unsigned char dsm[];

    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int nw = (int)(blockDim.x >> 5);
    const int C = a.C, V = a.V, Kmax = a.Kmax, KW = a.kw;
    const uint32_t rank = cluster_ctarank();
    const int n_clusters = (int)(gridDim.x / (unsigned)C);
    const int cid = (int)(blockIdx.x / (unsigned)C);   // this cluster: ticket cid first
    // SPLIT: this warp's half (hv) and its place in it (wv); nwv warps of a
    // CTA walk together
    const bool half = SPLIT && cid >= n_clusters - a.split_clusters;
    const int nwv = half ? (nw >> 1) : nw;
    const int hv = half ? w / nwv : 0;
    const int wv = half ? w - hv * nwv : w;
    const int P = C * nwv;   // warps per row
    const int g = (int)rank * nwv + wv;   // this warp's range of the row
    const int c_lo = range_lo(g, a.nchunks, P);
    const int kwm = range_lo(g + 1, a.nchunks, P) - c_lo;   // chunks in range
    const int e0 = c_lo * CH;                               // first element of the range
    const int n_el = max(0, min(e0 + kwm * CH, V) - e0);
    const SweepLayout L = sweep_layout(nw, cta_chunks(a.nchunks, C), KW, CH * (int)sizeof(T), C * nw);

    // the slice's place in the CTA's target and draft regions (a half's
    // slices: in the target region for half 0, the draft region for half 1)
    const size_t off = (size_t)(c_lo - range_lo((int)rank * nwv, a.nchunks, P)) * CH;
    T* slot_t = reinterpret_cast<T*>(dsm + (hv ? L.region_bytes : 0)) + off;
    T* slot_d = half ? slot_t : reinterpret_cast<T*>(dsm + L.region_bytes) + off;
    const uint32_t bar = smem_addr(dsm + L.bars + 8 * (size_t)w);
    // a split cluster never takes a sampling row: half 1 exchanges its rows on
    // the residual exchange's barriers and buffers, and keeps its claims in
    // the (unused) strip-partial area
    uint64_t* xbar = reinterpret_cast<uint64_t*>(dsm + (hv ? L.xbar2 : L.xbar));
    uint64_t* xbar2 = reinterpret_cast<uint64_t*>(dsm + L.xbar2);
    float4* xbuf = reinterpret_cast<float4*>(dsm + (hv ? L.xbuf2 : L.xbuf));   // [2][P]
    float2* xbuf2 = reinterpret_cast<float2*>(dsm + L.xbuf2);                  // [2][P]
    int2* xclaim = reinterpret_cast<int2*>(dsm + (hv ? L.stats + 16 : L.xclaim));   // [2]
    const uint32_t xbarc = smem_addr(dsm + (hv ? L.stats : L.xbarc));
    int* first = reinterpret_cast<int*>(dsm + (hv ? L.stats + 8 : L.first));
    float* stats = reinterpret_cast<float*>(dsm + L.stats) + (size_t)w * KW * 16;   // [kw][NV][4]
    // a half's strip sums, one per strip ([2 kw][NV]: a half's ranges are at
    // most twice as long), after half 1's claim slots (32 bytes): 32 + nw *
    // 2 kw * NV * 4 bytes fit in the area's nw * kw * 64 at NV = 4
    float* hstats = reinterpret_cast<float*>(dsm + L.stats + 32) + (size_t)w * 2 * KW * NV;

    // ---- set-up: barriers; -inf past V in this warp's range (copies never
    // write there); the cluster's first unit from rank 0 ----
    if (lane == 0) {
        mbar_init(bar, 1);
        if (w == 0) {
            mbar_init(smem_addr(&xbar[0]), 1);
            mbar_init(smem_addr(&xbar[1]), 1);
            mbar_init(smem_addr(&xbar2[0]), 1);
            mbar_init(smem_addr(&xbar2[1]), 1);
            mbar_init(xbarc, 1);
        }
        if (half && wv == 0 && hv == 1)   // half 1's claim barrier
            mbar_init(xbarc, 1);
        fence_mbar_init();
    }
    for (int j = n_el + lane; j < kwm * CH; j += 32) {
        EL::set_neg_inf(slot_t + j);
        EL::set_neg_inf(slot_d + j);
    }
    // this CTA's slice of the header's K and order, into the workspace
    if (a.copy_hdr) {
        const int per = (a.B + (int)gridDim.x - 1) / (int)gridDim.x;
        const int lo = (int)blockIdx.x * per, hi = min(a.B, lo + per);
        for (int j = lo + (int)threadIdx.x; j < hi; j += (int)blockDim.x) {
            a.K_dev[j] = __ldg(a.K + j);
            a.order_dev[j] = __ldg(a.order + j);
        }
    }
    __syncthreads();
    if (a.copy_hdr && threadIdx.x == 0) {
        __threadfence();   // the slice before the count that publishes it
        atomicAdd(a.ready, 1);
    }
    cluster_arrive();   // every CTA's barriers exist before any peer signals them
    cluster_wait();

    // ---- per-warp schedule state (the same in every warp of the walker) ----
    // first-wave slot and ticket: cluster cid; with SPLIT, the sampling queue's
    // tickets 0 .. n_full - 1 go to the whole clusters and the greedy queue's
    // first 2 split_clusters tickets to the halves
    const int n_full = n_clusters - (SPLIT ? a.split_clusters : 0);
    const int fslot = half ? n_full + 2 * (cid - n_full) + hv : cid;
    const int t0 = half ? a.split_ns + 2 * (cid - n_full) + hv : cid;
    bool hdr_dev = false;   // the header's device copy is complete (sticky)
    const int u0 = fslot < kFirstUnits ? a.first_b[fslot] : ticket_unit(a, t0, hdr_dev);
    bool active = u0 >= 0 && u0 < a.B;
    int spare = -1;
    UnitPos spare_pos{0, 0, 0.0f};
    bool exhausted = false;
    // A cluster claims its next sequence a row ahead (hiding the claim's
    // latency) only while at least two waves of tickets remain; nearer the
    // end it claims when it finishes a sequence, so that the last sequences
    // go to the clusters that are free first.  (The ticket of a row-ahead
    // claim is taken when the previous row is issued; see claim_next.)
    int last_t = t0;         // the ticket of the walker's latest claim
    uint32_t kc = 0;         // claims made between sequences (xbarc phase)
    bool broken = false;     // a slot wait gave up: no more copies, rows poisoned
    bool xbroken = false;    // an exchange wait gave up: leave the loop
    bool drawn = false;      // the current sequence's outputs are written
    Row row = make_row(a, 0, 0, 0, 0.0f, 0, 0);
    SeqVals cur_sv{0, 0.0f}, spare_sv{0, 0.0f};   // the current and the spare sequence's
    if (active) {
        const UnitPos p0 = first_unit_pos(a, fslot, u0, hdr_dev);
        row = make_row(a, 0, p0.b, p0.Kb, p0.T, p0.tb, p0.db);
        cur_sv = seq_vals(a, u0, lane);
        if (half)
            row = no_draft_only(a, row, lane);
    }
    Tok tk{0, 0.0f, 0u, 0u, 0};       // lane 0
    float uf = 0.0f;                  // lane 0: the sequence's final uniform
    int ticket = -1;                  // rank 0, warp 0, lane 0
    uint32_t uses = 0;                // completed slot fills (mbarrier phase)
    bool pending = false;             // a slot fill is in flight
    uint32_t k2 = 0;                  // residual exchanges so far
    const long long max_rows = (long long)a.B * (Kmax + 1) + 2;

    const T* tgt = static_cast<const T*>(a.tgt);
    const T* drf = static_cast<const T*>(a.drf);
    const bool writer = rank == 0 && wv == 0;   // writes per-row results and short outputs
    // (wv == 0: the warp of each CTA that arms its walker's exchange barriers)
    // the walker's claims: whole clusters take the sampling queue, then the
    // greedy one; halves the greedy one
    auto claim = [&]() -> int {
        if constexpr (SPLIT) {
            if (!half) {
                const int t = atomicAdd(a.next_unit, 1) + n_full;
                if (t < a.split_ns)
                    return t;
            }
            return a.split_ns + atomicAdd(a.next_unit_g, 1) + 2 * a.split_clusters;
        } else {
            return claim_ticket(a, n_clusters);
        }
    };

    // copies of this warp's range of row r into the slot (whole warp)
    auto issue = [&](const Row& r) {
        if (!(r.flags & kFUsable) || broken || n_el <= 0)
            return;
        const bool ld = (r.flags & kFDraft) != 0;
        const T* tr = tgt + ((size_t)r.tb + r.i) * (size_t)V + e0;
        const T* dr = ld ? drf + ((size_t)r.db + r.i) * (size_t)V + e0 : nullptr;
        const int nb = a.aligned ? ((n_el * (int)sizeof(T)) & ~15) / (int)sizeof(T) : 0;
        if constexpr (HOST) {
            // logits in device-mapped host memory: 16-byte loads (the bulk-copy
            // engine is not used on host memory), eight in flight per lane,
            // stored to the slot (lane l stores the vectors it reads in the
            // pass); the rest one element at a time; then a plain arrival on
            // the slot barrier
            const int nvec = nb * (int)sizeof(T) / 16;
            for (int arr = 0; arr < (ld ? 2 : 1); ++arr) {
                const uint4* src = reinterpret_cast<const uint4*>(arr ? dr : tr);
                uint4* dst = reinterpret_cast<uint4*>(arr ? slot_d : slot_t);
                for (int j0 = 0; j0 < nvec; j0 += 8 * 32) {
                    uint4 x[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const int j = j0 + u * 32 + lane;
                        if (j < nvec)
                            x[u] = src[j];
                    }
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const int j = j0 + u * 32 + lane;
                        if (j < nvec)
                            dst[j] = x[u];
                    }
                }
            }
            for (int j = nb + lane; j < n_el; j += 32) {
                EL::copy(slot_t + j, tr + j);
                if (ld)
                    EL::copy(slot_d + j, dr + j);
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(bar);
            pending = true;
            return;
        }
        if (lane == 0) {
            const uint32_t bytes = (uint32_t)nb * (uint32_t)sizeof(T);
            const uint32_t tx = bytes * (ld ? 2u : 1u);
            if (tx) {
                fence_proxy_async();
                mbar_arrive_expect_tx(bar, tx);
                // each row is read once: its lines go first from L2, ahead
                // of prefetched rows and the small per-row arrays
                const uint64_t pol = l2_evict_first_policy();
                bulk_copy_g2s_hint(smem_addr(slot_t), tr, bytes, bar, pol);
                if (ld)
                    bulk_copy_g2s_hint(smem_addr(slot_d), dr, bytes, bar, pol);
            } else {
                mbar_arrive(bar);
            }
        }
        for (int j = nb + lane; j < n_el; j += 32) {
            EL::copy(slot_t + j, tr + j);
            if (ld)
                EL::copy(slot_d + j, dr + j);
        }
        pending = true;
    };
    // wait for the slot fill (whole warp); false if any lane gave up (at
    // once when the caller asked for expired waits, to test this path)
    const uint32_t slot_spins = a.expire_waits ? 0u : kWaitSpins;
    auto wait_slot = [&]() -> bool {
        const bool ok = mbar_wait_bounded(bar, uses & 1u, slot_spins);
        const bool all = !__any_sync(kFull, !ok);
        if (all) {
            pending = false;
            ++uses;
        }
        __syncwarp();
        return all;
    };
    // The spare sequence's first row is read whatever the current rows
    // decide, so this warp's range of it is brought into L2 as soon as the
    // spare is known: its target row at once, its draft row (sampling
    // sequences with a tested row only) once the spare's K and T have loaded.
    bool pf_draft = false;   // the spare's draft row is still to prefetch
    const int nb_pf = a.aligned ? ((n_el * (int)sizeof(T)) & ~15) / (int)sizeof(T) : 0;
    auto prefetch_target = [&](int trow) {
        if (lane == 0 && nb_pf > 0 && !HOST)
            bulk_prefetch_l2(tgt + (size_t)trow * (size_t)V + e0, (uint32_t)nb_pf * (uint32_t)sizeof(T));
    };
    auto prefetch_draft = [&]() {   // (and the target's, packed: its row had to load)
        if (spare < 0)
            return;
        if (a.packed)
            prefetch_target(spare_pos.tb);
        if (lane == 0 && nb_pf > 0 && !HOST && a.has_draft && spare_pos.Kb > 0 && spare_pos.T != 0.0f)
            bulk_prefetch_l2(drf + (size_t)spare_pos.db * (size_t)V + e0, (uint32_t)nb_pf * (uint32_t)sizeof(T));
    };

    // per-warp counters (lane 0), added to the call's sv_stats at exit
    uint32_t c_seq = 0, c_inv = 0, c_test = 0, c_acc = 0, c_commit = 0, c_tie = 0;

    // outputs of the current sequence b (whole warp): draft tokens before n
    // (n <= 32, from the sequence's registers), `token` at n, -1 after.  Each
    // sequence's outputs are written exactly once, so its KV length is
    // committed here too.
    auto write_outputs = [&](int b, int n, int token, int seq_tok) {
        const bool bad = token < 0;
        int32_t* orow = a.out_tok + (size_t)b * (Kmax + 1);
        for (int j = lane; j <= Kmax; j += 32)
            orow[j] = bad ? -1 : (j < n ? seq_tok : (j == n ? token : -1));
        if (lane == 0) {
            a.out_n[b] = bad ? -1 : n;
            if (a.want_final)
                a.final_row[b] = bad ? -1 : n;
            if (a.want_kv && !bad)
                a.kv_len[b] += n + 1;
            if (bad) {
                ++c_inv;
            } else {
                ++c_seq;
                c_commit += (uint32_t)n + 1u;
            }
        }
    };

    // A cluster claims its next sequence a row ahead.  The ticket (an atomic
    // on the claim counter) is taken when the row that needs it is issued,
    // one row before its order lookup: taken at the top of that row, the
    // lookup's address waited on the atomic's round trip and the claiming
    // warp started its pass about a microsecond after the others, holding
    // up every row that carried a claim.  It claims ahead only while two
    // waves of its queue remain (with SPLIT: the sampling queue for a whole
    // cluster still taking from it, else the greedy queue, which every walker
    // takes from in the end; a whole cluster that kept claiming ahead up to
    // the end of the sampling queue made workload 4 1.2% slower).
    auto ahead_ok = [&](int t) -> bool {
        if constexpr (SPLIT) {
            if (!half && t < a.split_ns)
                return (long long)t + 2LL * n_full < (long long)a.split_ns;
            return (long long)t + 2LL * (n_full + 2 * a.split_clusters) < (long long)a.B;
        } else {
            return (long long)t + 2LL * n_clusters < (long long)a.B;
        }
    };
    bool claim_next = spare < 0 && !exhausted && ahead_ok(last_t);
    if (active) {
        issue(row);
        if (writer && lane == 0 && claim_next)
            ticket = claim();
        tk = tok_of(a, row, cur_sv);
        if (lane == 0) {
            tok_logits<T>(a, row, tk);
            uf = final_uniform(a, row);
        }
    }

    for (long long k = 0; active && k < max_rows; ++k) {
        const int p = (int)(k & 1);
        const uint32_t xpar = (uint32_t)((k >> 1) & 1);
        const bool greedy = (row.flags & kFGreedy) != 0;
        const bool test = (row.flags & kFTest) != 0;
        const bool draft = (row.flags & kFDraft) != 0;
        const bool usable = (row.flags & kFUsable) != 0;
        const float c = (usable && !greedy) ? log2e_over(row.T) : 0.0f;
        const bool want_claim = claim_next;   // this row carries a claim (ticket taken)
        if (wv == 0 && lane == 0)
            mbar_arrive_expect_tx(smem_addr(&xbar[p]), (uint32_t)P * 16u + (want_claim ? 8u : 0u));

        // ---- the slice, then the proposal's logits and the claim's sequence ----
        bool have = false;
        if (pending) {
            have = wait_slot();
            if (!have)
                broken = true;
        }
        int claimed = -1;   // the order lookup now, its checks after the pass
        if (writer && lane == 0 && want_claim)
            claimed = ticket_load(a, ticket, hdr_dev);

        // ---- one pass over this warp's slice ----
        const float ref_t = EL::widen(__shfl_sync(kFull, tk.lt, 0));
        const float ref_d = EL::widen(__shfl_sync(kFull, tk.ld, 0));
        const bool ref_ok = __shfl_sync(kFull, tk.ok, 0) && isfinite(ref_t) && isfinite(ref_d);
        float4 part = make_float4(-INFINITY, __int_as_float(INT_MAX), -INFINITY, 0.0f);
        if (greedy) {
            float gm = -INFINITY;
            int gi = INT_MAX;
            if (have) {
                // the lane's maximum and the first chunk holding it (selects,
                // no branch: a search inside the loop ran whenever any lane's
                // maximum grew, which is nearly every chunk), then one search
                // of that chunk for the lowest element holding it
                int gj = -1;
#pragma unroll 1
                for (int j = 0; j < kwm; ++j) {
                    uint4 tv[NV];
                    load_chunk<T, NV>(slot_t + (size_t)j * CH, lane, tv);
                    const float cm = LN::max(tv);
                    const bool up = cm > gm;   // strictly greater: an earlier chunk keeps a tie
                    gj = up ? j : gj;
                    gm = up ? cm : (cm != cm ? cm : gm);
                }
                if (gj >= 0 && gm == gm) {
                    uint4 tv[NV];
                    load_chunk<T, NV>(slot_t + (size_t)gj * CH, lane, tv);
                    const int gbase = e0 + gj * CH;
#pragma unroll
                    for (int e = NV * E - 1; e >= 0; --e)   // the lowest match wins
                        if (LN::elem(tv, e) == gm)
                            gi = gbase + ((e / E) * 32 + lane) * E + (e % E);
                }
            }
            const float m = warp_max_nan(gm);
            const int gidx = __reduce_min_sync(kFull, gm == m ? gi : INT_MAX);
            part = make_float4(m, __int_as_float(gidx), -INFINITY, 0.0f);
        } else if (test && !(row.flags & kFMaxRef) && ref_ok) {
            // weights against the proposal's logits: one sweep, and every
            // warp's sums share the reference, so the partials simply add
            float st = 0.0f, sd = 0.0f;
            if (have) {
#pragma unroll 1
                for (int j = 0; j < kwm; ++j) {
                    uint4 v[NV];
                    load_chunk<T, NV>(slot_t + (size_t)j * CH, lane, v);
                    st += LN::exp_sum(v, ref_t, c);
                    load_chunk<T, NV>(slot_d + (size_t)j * CH, lane, v);
                    sd += LN::exp_sum(v, ref_d, c);
                }
            }
            // an overflowed weight makes the warp's sum +inf (the compensated
            // sum would turn it into NaN, which means unusable input)
            sum_or_special2(st, sd);
            part = make_float4(ref_t, st, ref_d, sd);
        } else if (test) {
            // weights against the running lane maxima
            float mt = -INFINITY, st = 0.0f, md = -INFINITY, sd = 0.0f;
            if (have) {
#pragma unroll 1
                for (int j = 0; j < kwm; ++j) {
                    uint4 tv[NV], dv[NV];
                    load_chunk<T, NV>(slot_t + (size_t)j * CH, lane, tv);
                    load_chunk<T, NV>(slot_d + (size_t)j * CH, lane, dv);
                    const float nt = max_nan(mt, LN::max(tv));
                    if (nt != mt) {   // the lane max grew (or turned NaN): rescale the sum
                        st = mt == -INFINITY ? 0.0f : st * weight(mt, nt, c);
                        mt = nt;
                    }
                    st += LN::exp_sum(tv, mt == -INFINITY ? 0.0f : mt, c);
                    const float nd = max_nan(md, LN::max(dv));
                    if (nd != md) {
                        sd = md == -INFINITY ? 0.0f : sd * weight(md, nd, c);
                        md = nd;
                    }
                    sd += LN::exp_sum(dv, md == -INFINITY ? 0.0f : md, c);
                }
            }
            float m1, S1, m2, S2;
            combine_ms2(mt, st, md, sd, c, m1, S1, m2, S2);
            part = make_float4(m1, S1, m2, S2);
        } else {
            // bonus row: the warp's maximum, then per-strip sums against it
            // (kept for the draw)
            float mm = -INFINITY, acc = 0.0f, cmp = 0.0f;
            if (have) {
                float lm = -INFINITY;
#pragma unroll 1
                for (int j = 0; j < kwm; ++j) {
                    uint4 tv[NV];
                    load_chunk<T, NV>(slot_t + (size_t)j * CH, lane, tv);
                    lm = max_nan(lm, LN::max(tv));
                }
                mm = warp_max_nan(lm);
                const float mu = mm == -INFINITY ? 0.0f : mm;
#pragma unroll 1
                for (int j = 0; j < kwm; ++j) {
                    uint4 tv[NV];
                    load_chunk<T, NV>(slot_t + (size_t)j * CH, lane, tv);
                    float sv[NV];
                    LN::exp_strips(tv, mu, c, sv);
                    if (half)
                        strip_partials<NV, true>(sv, lane, hstats + (size_t)j * NV);
                    else
                        strip_partials<NV>(sv, lane, stats + (size_t)j * NV * 4);
                    float v = 0.0f;
#pragma unroll
                    for (int k = 0; k < NV; ++k)
                        v += sv[k];
                    float t, e;
                    two_sum(acc, v, t, e);
                    acc = t;
                    cmp += e;
                }
                __syncwarp();
            }
            part = make_float4(mm, sum_or_special(acc + cmp), -INFINITY, 0.0f);
        }
        if (broken)
            part.x = NAN;   // poisons the row in every warp of the cluster

        // ---- exchange: this warp's partial to every CTA of the cluster ----
        if (writer && lane == 0 && want_claim)
            claimed = ticket_check(a, ticket, claimed);
        const int claimed_b = __shfl_sync(kFull, claimed, 0);
        const int claimed_t = __shfl_sync(kFull, ticket, 0);
        if (lane < C) {
            const uint32_t rb = map_to_rank(smem_addr(&xbar[p]), (uint32_t)lane);
            st_async_v4(map_to_rank(smem_addr(&xbuf[p * P + g]), (uint32_t)lane), part, rb);
            if (writer && want_claim)
                st_async_v2(map_to_rank(smem_addr(&xclaim[p]), (uint32_t)lane),
                            make_float2(__int_as_float(claimed_b), __int_as_float(claimed_t)), rb);
        }
        if (pf_draft) {   // the spare's K and T have long loaded
            prefetch_draft();
            pf_draft = false;
        }
        if (!mbar_wait_bounded(smem_addr(&xbar[p]), xpar, kWaitSpins))
            xbroken = true;
        if (__any_sync(kFull, xbroken))
            break;

        // ---- combine all partials and decide (every warp alike) ----
        // lane j holds the partials of warps j and j + 32
        const float4 xnone = make_float4(-INFINITY, __int_as_float(INT_MAX), -INFINITY, 0.0f);
        const bool has = lane < P, has2 = WIDE && lane + 32 < P;
        const float4 xv = has ? xbuf[p * P + lane] : xnone;
        const float4 xw = has2 ? xbuf[p * P + lane + 32] : xnone;
        const TokF tkb = shfl_tok<T>(tk);
        const size_t pos = (size_t)row.b * Kmax + row.i;   // diagnostics index (test rows)
        int dec = kDecInvalid;
        bool redo = false;
        bool near_tie = false;   // the uniform within 1e-6 of p/q (sampling tests)
        int gtok = -1;
        float m_t = 0.0f, m_d = 0.0f, inv_st = 0.0f, inv_sd = 0.0f;
        bool row_ok = false;
        if (greedy) {
            m_t = warp_max_nan(WIDE ? max_nan(xv.x, xw.x) : xv.x);
            const int i1 = (has && xv.x == m_t) ? __float_as_int(xv.y) : INT_MAX;
            const int i2 = (has2 && xw.x == m_t) ? __float_as_int(xw.y) : INT_MAX;
            gtok = __reduce_min_sync(kFull, min(i1, i2));
            row_ok = usable && tkb.ok && isfinite(m_t) && gtok < V;
            dec = !row_ok ? kDecInvalid : (test ? (tkb.x == gtok ? kDecAccept : kDecReject) : kDecBonus);
            if (writer && lane == 0 && test && a.want_pq) {
                a.p_x[pos] = NAN;
                a.q_x[pos] = NAN;
            }
        } else {
            float St, Sd;
            // weights against the proposal's logits that overflowed: the row
            // is weighed again against its maxima (same data, same result)
            const bool any_inf = __any_sync(kFull, (has && (isinf(xv.y) || isinf(xv.w))) ||
                                                       (has2 && (isinf(xw.y) || isinf(xw.w))));
            const bool any_nan =
                __any_sync(kFull, (has && (isnan(xv.x) || isnan(xv.y) || isnan(xv.z) || isnan(xv.w))) ||
                                      (has2 && (isnan(xw.x) || isnan(xw.y) || isnan(xw.z) || isnan(xw.w))));
            const bool refmode = test && !(row.flags & kFMaxRef) && ref_ok;
            redo = refmode && !broken && any_inf && !any_nan;
            if (refmode) {
                // every warp weighed against the proposal's logits: the
                // partials share that reference and simply add
                m_t = ref_t;
                m_d = ref_d;
                St = has ? xv.y : 0.0f;
                Sd = has ? xv.w : 0.0f;
                if (has2) {
                    St += xw.y;
                    Sd += xw.w;
                }
                warp_sum_comp2(St, Sd);
            } else {
                float ma = xv.x, sa = xv.y, mb = xv.z, sb = xv.w;
                if (has2) {
                    merge_ms(ma, sa, xw.x, xw.y, c);
                    merge_ms(mb, sb, xw.z, xw.w, c);
                }
                combine_ms2(ma, sa, mb, sb, c, m_t, St, m_d, Sd);
            }
            row_ok = !redo && !any_nan && usable && tkb.ok && isfinite(m_t) && St > 0.0f && isfinite(St) &&
                     (!draft || (isfinite(m_d) && Sd > 0.0f && isfinite(Sd)));
            bool accept = false;
            if (test && row_ok) {
                if (refmode) {
                    // p(x) = w_t(x) / S_t and q(x) = w_d(x) / S_d, both weights
                    // taken against themselves (exp2(0) = 1): u < min(1, p/q)
                    // reads u S_t < S_d, with no exponential or division
                    accept = __fmul_rn(tkb.u, St) < Sd;
                    near_tie = fabsf(__fmaf_rn(tkb.u, St, -Sd)) < 1e-6f * St;
                } else {
                    const float px = __fmul_rn(weight(tkb.lt, m_t, c), __frcp_rn(St));
                    const float qx = __fmul_rn(weight(tkb.ld, m_d, c), __frcp_rn(Sd));
                    accept = __fmul_rn(tkb.u, qx) < px;   // u < min(1, p/q) without a division
                    near_tie = fabsf(__fmaf_rn(tkb.u, qx, -px)) < 1e-6f * qx;
                }
            }
            dec = redo ? kDecRedo
                       : (!row_ok ? kDecInvalid : (test ? (accept ? kDecAccept : kDecReject) : kDecBonus));
            // the inverse sums, where the residual pass or the diagnostics need them
            if (row_ok && (dec == kDecReject || !a.early_exit || a.want_pq)) {
                inv_st = __frcp_rn(St);
                inv_sd = draft ? __frcp_rn(Sd) : 0.0f;
            }
            if (writer && lane == 0 && test && a.want_pq && !redo) {
                a.p_x[pos] = row_ok ? __fmul_rn(weight(tkb.lt, m_t, c), inv_st) : NAN;
                a.q_x[pos] = row_ok ? __fmul_rn(weight(tkb.ld, m_d, c), inv_sd) : NAN;
            }
        }
        // counters: the tested positions the method walks (up to the stop)
        if (writer && lane == 0 && a.want_stats && test && !drawn && (dec == kDecAccept || dec == kDecReject)) {
            ++c_test;
            c_acc += dec == kDecAccept ? 1u : 0u;
            c_tie += near_tie ? 1u : 0u;
        }
        if (want_claim) {
            const int2 clv = xclaim[p];
            const int cl = clv.x;
            spare = (cl >= 0 && cl < a.B) ? cl : -1;
            exhausted = spare < 0;
            if (spare >= 0)
                last_t = clv.y;
            if (spare >= 0) {
                spare_pos = unit_pos(a, spare, hdr_dev);   // loads now, used when the unit starts
                spare_sv = seq_vals(a, spare, lane);
                if (!a.packed)
                    prefetch_target(spare * (Kmax + 1));
                pf_draft = true;
            }
        }

        // ---- residual pass: rows that may be drawn from (resident slice) ----
        const bool resid_pass = !greedy && test && draft && row_ok && !broken &&
                                (dec == kDecReject || !a.early_exit);
        float S_R = 0.0f;
        float2 wtot = make_float2(0.0f, 0.0f);    // lane j: warp j's (residual, p) totals
        float2 wtot2 = make_float2(0.0f, 0.0f);   // and warp j + 32's
        if (resid_pass) {
            float rs_s = 0.0f, rs_c = 0.0f, ps_s = 0.0f, ps_c = 0.0f;
#pragma unroll 1
            for (int j = 0; j < kwm; ++j) {
                uint4 tv[NV], dv[NV];
                load_chunk<T, NV>(slot_t + (size_t)j * CH, lane, tv);
                load_chunk<T, NV>(slot_d + (size_t)j * CH, lane, dv);
                float rsv[NV], ps;
                LN::resid_strips(tv, dv, m_t, inv_st, m_d, inv_sd, c, rsv, ps);
                strip_partials<NV>(rsv, lane, stats + (size_t)j * NV * 4);
                float rs = 0.0f;
#pragma unroll
                for (int k = 0; k < NV; ++k)
                    rs += rsv[k];
                float t, e;
                two_sum(rs_s, rs, t, e);
                rs_s = t;
                rs_c += e;
                two_sum(ps_s, ps, t, e);
                ps_s = t;
                ps_c += e;
            }
            __syncwarp();
            rs_s += rs_c;
            ps_s += ps_c;
            warp_sum_comp2(rs_s, ps_s);
            rs_c = 0.0f;
            ps_c = 0.0f;
            const int p2 = (int)(k2 & 1);
            const uint32_t par2 = (k2 >> 1) & 1u;
            ++k2;
            if (w == 0 && lane == 0)
                mbar_arrive_expect_tx(smem_addr(&xbar2[p2]), (uint32_t)P * 8u);
            if (lane < C) {
                const uint32_t rb = map_to_rank(smem_addr(&xbar2[p2]), (uint32_t)lane);
                const uint32_t dst = map_to_rank(smem_addr(&xbuf2[p2 * P + g]), (uint32_t)lane);
                st_async_v2(dst, make_float2(rs_s + rs_c, ps_s + ps_c), rb);
            }
            if (pf_draft) {
                prefetch_draft();
                pf_draft = false;
            }
            if (!mbar_wait_bounded(smem_addr(&xbar2[p2]), par2, kWaitSpins))
                xbroken = true;
            if (__any_sync(kFull, xbroken))
                break;
            wtot = has ? xbuf2[p2 * P + lane] : make_float2(0.0f, 0.0f);
            wtot2 = has2 ? xbuf2[p2 * P + lane + 32] : make_float2(0.0f, 0.0f);
            S_R = warp_sum_comp(WIDE ? wtot.x + wtot2.x : wtot.x);
        }
        if (writer && lane == 0 && test && a.want_resid && !redo)
            a.resid[pos] = resid_pass ? S_R : NAN;

        // ---- the sequence's final row: its token and outputs ----
        if (!drawn && dec != kDecAccept && !redo) {
            drawn = true;
            const int n = row.i;
            const float ufb = __shfl_sync(kFull, uf, 0);
            if (dec == kDecInvalid || (!greedy && !(ufb >= 0.0f && ufb < 1.0f))) {
                if (writer)
                    write_outputs(row.b, n, -1, cur_sv.tok);
            } else if (greedy) {
                if (writer)
                    write_outputs(row.b, n, gtok, cur_sv.tok);
            } else {
                // per-warp masses of the distribution drawn from: the residual
                // (zero residual mass: p of the same row), or p at the bonus row
                const bool bonus = dec == kDecBonus;
                const bool use_r = !bonus && S_R > 0.0f;
                float Wj = 0.0f, Wj2 = 0.0f;   // lane j: the masses of warps j and j + 32
                if (has)
                    Wj = bonus ? (xv.x == -INFINITY ? 0.0f : xv.y * weight(xv.x, m_t, c))
                               : (use_r ? wtot.x : wtot.y);
                if (has2)
                    Wj2 = bonus ? (xw.x == -INFINITY ? 0.0f : xw.y * weight(xw.x, m_t, c))
                                : (use_r ? wtot2.x : wtot2.y);
                // the warp whose range holds u * S, and the mass left inside it
                float t = 0.0f, S_draw = 0.0f;   // the point and the total mass
                bool beyond = false;
                int owner = -1;
                if constexpr (WIDE) {
                    const float S = warp_sum_comp(Wj + Wj2);
                    if (S > 0.0f && isfinite(S)) {
                        S_draw = S;
                        t = ufb * S;
                        owner = select_cdf(P, [&](int j) { return j < 32 ? Wj : Wj2; }, t, beyond, lane);
                    }
                } else {   // one mass per lane: one compensated scan
                    float s, cc;
                    warp_incl_scan_comp(Wj, lane, s, cc);
                    const float S = __shfl_sync(kFull, s, 31) + __shfl_sync(kFull, cc, 31);
                    if (S > 0.0f && isfinite(S)) {
                        S_draw = S;
                        t = ufb * S;
                        const unsigned hit = __ballot_sync(kFull, lane < P && Wj > 0.0f && t < s + cc);
                        if (hit) {
                            owner = __ffs(hit) - 1;
                            const float os = __shfl_sync(kFull, s, owner);
                            const float oc = __shfl_sync(kFull, cc, owner);
                            const float ow = __shfl_sync(kFull, Wj, owner);
                            t = t - ((os - ow) + oc);
                        } else {
                            const unsigned posm = __ballot_sync(kFull, lane < P && Wj > 0.0f);
                            owner = posm ? 31 - __clz(posm) : -1;
                            beyond = true;
                        }
                    }
                }
                if (owner < 0) {
                    if (writer)
                        write_outputs(row.b, n, -1, cur_sv.tok);
                } else if (owner == g) {
                    // this warp holds the token: its chunk, the strip, then the
                    // element.  Zero residual mass: p's strip sums are made
                    // first (the residual pass kept only p's warp totals).
                    if (!bonus && !use_r) {
#pragma unroll 1
                        for (int j = 0; j < kwm; ++j) {
                            uint4 tv[NV];
                            load_chunk<T, NV>(slot_t + (size_t)j * CH, lane, tv);
                            float sv[NV];
                            LN::exp_strips(tv, m_t, c, sv);
                            strip_partials<NV>(sv, lane, stats + (size_t)j * NV * 4);
                        }
                        __syncwarp();
                    }
                    // masses: sums of the strips' four partials (the bonus pass
                    // summed against this warp's own maximum, that of partial g)
                    const float own_m = __shfl_sync(kFull, (WIDE && g >= 32) ? xw.x : xv.x, g & 31);
                    const float wscale = bonus ? (own_m == -INFINITY ? 0.0f : weight(own_m, m_t, c)) : 1.0f;
                    // strips in index order: chunk j's strip k is entry j * NV + k
                    // (a half keeps each strip's sum alone)
                    auto strip_mass = [&](int q) -> float {
                        if (half)
                            return hstats[q] * wscale;
                        const float4 v = *reinterpret_cast<const float4*>(stats + (size_t)q * 4);
                        return ((v.x + v.y) + (v.z + v.w)) * wscale;
                    };
                    float tc = t;
                    int token = -1;
                    const int js = select_cdf(kwm * NV, strip_mass, tc, beyond, lane);
                    if (js >= 0) {
                        const int jc = js / NV, ks = js % NV;
                        {
                            const uint4* vt = reinterpret_cast<const uint4*>(slot_t + (size_t)jc * CH);
                            const uint4* vd = reinterpret_cast<const uint4*>(slot_d + (size_t)jc * CH);
                            const uint4 tk = vt[ks * 32 + lane];
                            const uint4 dk = use_r ? vd[ks * 32 + lane] : tk;
                            bool near = false;
                            const int ce = pick_in_strip<T, NV, false>(tk, dk, use_r, m_t, inv_st, m_d, inv_sd, c,
                                                                       tc, beyond, lane, 0.0f, near);
                            if (ce >= 0)
                                token = e0 + jc * CH + ks * 32 * E + ce;
                            if (a.want_stats && token >= 0 && token < V &&
                                draw_is_near<T, NV>(tk, dk, use_r, m_t, inv_st, m_d, inv_sd, c, tc, beyond, lane,
                                                    1e-6f * S_draw) && lane == 0)
                                atomicAdd(a.stats + 6, 1ull);
                        }
                    }
                    write_outputs(row.b, n, (token >= 0 && token < V) ? token : -1, cur_sv.tok);
                }
            }
        }

        // ---- the cluster's next row (the same decision in every warp) ----
        const bool valid = dec == kDecAccept || dec == kDecReject;
        const bool cont = redo || (row.i < row.Kb && (dec == kDecAccept || (!a.early_exit && valid)));
        if (!cont && writer && (a.want_pq || a.want_resid)) {
            // positions this sequence does not reach carry NaN diagnostics
            for (int i = (test ? row.i + 1 : row.i) + lane; i < Kmax; i += 32) {
                const size_t q = (size_t)row.b * Kmax + i;
                if (a.want_pq) {
                    a.p_x[q] = NAN;
                    a.q_x[q] = NAN;
                }
                if (a.want_resid)
                    a.resid[q] = NAN;
            }
        }
        if (redo) {
            row.flags |= kFMaxRef;   // the same row again
        } else if (cont) {
            row = make_row(a, row.i + 1, row.b, row.Kb, row.T, row.tb, row.db);
        } else {
            if (spare < 0 && !exhausted) {
                // claim now: rank 0's writer takes a ticket and sends the
                // sequence to every CTA (st.async onto each CTA's claim
                // mbarrier, bounded wait, as the row exchange)
                if (wv == 0 && lane == 0)
                    mbar_arrive_expect_tx(xbarc, 8u);
                int cb = -1, ct = -1;
                if (writer && lane == 0) {
                    ct = claim();
                    cb = ticket_unit(a, ct, hdr_dev);
                }
                cb = __shfl_sync(kFull, cb, 0);
                ct = __shfl_sync(kFull, ct, 0);
                if (writer && lane < C)
                    st_async_v2(map_to_rank(smem_addr(first), (uint32_t)lane),
                                make_float2(__int_as_float(cb), __int_as_float(ct)),
                                map_to_rank(xbarc, (uint32_t)lane));
                if (!mbar_wait_bounded(xbarc, kc & 1u, kWaitSpins))
                    xbroken = true;
                ++kc;
                if (__any_sync(kFull, xbroken))
                    break;
                const int nb = first[0];
                if (nb >= 0 && nb < a.B) {
                    spare = nb;
                    last_t = first[1];
                    spare_pos = unit_pos(a, nb, hdr_dev);
                    spare_sv = seq_vals(a, nb, lane);
                } else {
                    exhausted = true;
                }
            }
            if (spare < 0)
                break;
            row = make_row(a, 0, spare_pos.b, spare_pos.Kb, spare_pos.T, spare_pos.tb, spare_pos.db);
            if (half)
                row = no_draft_only(a, row, lane);
            cur_sv = spare_sv;
            spare = -1;
            drawn = false;
        }
        issue(row);   // copies first: the logit loads overlap with them
        claim_next = spare < 0 && !exhausted && ahead_ok(last_t);
        if (writer && lane == 0 && claim_next)
            ticket = claim();
        tk = tok_of(a, row, cur_sv);
        if (lane == 0) {
            tok_logits<T>(a, row, tk);
            if (!cont)
                uf = final_uniform(a, row);
        }
    }

    // ---- this warp's counters into the call's sv_stats ----
    if (a.want_stats && lane == 0) {
        const uint32_t cs[6] = {c_seq, c_inv, c_test, c_acc, c_commit, c_tie};
#pragma unroll
        for (int k = 0; k < 6; ++k)
            if (cs[k])
                atomicAdd(a.stats + k, (unsigned long long)cs[k]);
    }

    // ---- wind-down: a fill still in flight (only after a timeout), then
    // leave together, so that no CTA exits while a peer may still address it ----
    if (broken || xbroken) {
        if (lane == 0)
            atomicOr(a.err, kErrWaitTimeout);
        if (pending)
            (void)mbar_wait_bounded(bar, uses & 1u, kWaitSpins);
    }
    __syncwarp();
    cluster_arrive();
    cluster_wait();
}

}  // namespace sv
