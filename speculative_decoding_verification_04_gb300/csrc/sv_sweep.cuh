// sv_sweep.cuh -- the persistent vocabulary-sweep kernel.
//
// A grid of thread-block clusters (C CTAs each, as many as the device holds at
// once) works through the batch one row (sequence b, position i) at a time per
// cluster.  CTA r of a cluster owns the vocabulary chunks [r*ncpc, (r+1)*ncpc)
// of every row; warp w of the CTA owns every nw-th of those chunks and streams
// them through its own ring of R shared-memory stages (target and draft chunk
// per stage), filled by 1-D bulk copies (cp.async.bulk) that complete on one
// mbarrier per stage.  No two warps share a stage, so the steady state has no
// CTA-wide barrier at all.
//
// Schedule: a cluster walks one sequence's positions in order.  Row i+1 is
// read only once x_i has been accepted (the method's own early exit: rows after
// the first rejection are never read).  Fresh sequences come from one atomic
// claim per sequence (longest K first), made a row ahead by rank 0 and handed
// to the cluster with that row's exchange.  When there are fewer sequences
// than clusters, clusters claim single rows instead (all positions at once).
//
// Per row, each warp makes one pass over its chunks, from the stage straight
// into registers:
//   greedy row       lane max (packed bf16x2 / three-input fp32 max) and the
//                    lowest index holding it;
//   tested sampling  lane-online max and sum of exp2((l - m) log2(e)/T) of the
//   row              target and the draft row (rescaled when the lane max
//                    grows), in packed two-lane fp32 arithmetic;
//   bonus row        per-chunk (max, sum) of the target, kept for the draw.
// exchange  every warp pushes a 16-byte partial to every CTA of the cluster
//           with st.async, completing on the receiver's exchange mbarrier
//           (double-buffered by row parity);
// decide    every warp combines all C*nw partials (identical arithmetic, so
//           identical results) and decides u q(x) < p(x), or x == argmax at
//           temperature 0;
// residual  rejected rows (every tested row in verify-all mode): per-chunk
//           sums of max(0, p - q) and of p from the ring -- still resident
//           when the warp's chunks fit in it, read again through it otherwise.
// Results go to the workspace; sv_finalize draws the tokens.
#pragma once

#include "sv_common.cuh"

namespace sv {

constexpr int kMaxRing = 8;    // ring stages per warp
constexpr int kMaxParts = 32;  // C * nw partials per row: one per lane in the combine

// Dynamic shared memory of one CTA (host and device compute it alike).
struct SweepLayout {
    size_t stage_bytes;   // one stage: target chunk + draft chunk
    size_t bars;          // [nw][R] stage mbarriers
    size_t xbar;          // [2] exchange mbarriers
    size_t xbuf;          // [2][kMaxParts] float4 partials
    size_t xclaim;        // [2] int: unit claimed by rank 0 during the row
    size_t first;         // [2] int: first unit of the cluster (one used)
    size_t stats;         // [nw][kw] float2: per-chunk (max, sum) of bonus rows
    size_t total;
};

__host__ __device__ inline SweepLayout sweep_layout(int nw, int R, int chunk_bytes, int kw)
{
    SweepLayout L;
    L.stage_bytes = 2 * (size_t)chunk_bytes;
    L.bars = (size_t)nw * R * L.stage_bytes;
    L.xbar = L.bars + (size_t)nw * R * 8;
    L.xbuf = (L.xbar + 16 + 15) & ~(size_t)15;
    L.xclaim = L.xbuf + 2 * kMaxParts * 16;
    L.first = L.xclaim + 8;
    L.stats = L.first + 8;
    L.total = L.stats + (size_t)nw * kw * 8;
    return L;
}

// Row flags, from the sequence's K_b and T alone.
enum : int {
    kFGreedy = 1,   // T == 0
    kFTest = 2,     // i < K_b: a proposal is tested at this row
    kFDraft = 4,    // the draft row is read (tested sampling row)
    kFUsable = 8    // temperature usable and, if needed, draft logits supplied
};

struct Row {
    int i, b, Kb;
    float T;
    int flags;
};

__device__ __forceinline__ Row make_row(const Args& a, int i, int b, int Kb, float T)
{
    Row r;
    r.i = i;
    r.b = b;
    r.Kb = Kb;
    r.T = T;
    const int greedy = T == 0.0f ? kFGreedy : 0;
    const int test = i < Kb ? kFTest : 0;
    const int draft = (test && !greedy) ? kFDraft : 0;
    const int usable = (temperature_usable(T) && (!draft || a.has_draft != 0)) ? kFUsable : 0;
    r.flags = greedy | test | draft | usable;
    return r;
}

// What the decision needs besides the sums: the proposed token, its uniform
// and the two logits at the token.  Loaded by one lane a row ahead.
struct Tok {
    int x;
    float u, lt, ld;
    int ok;
};

template <typename T>
__device__ __forceinline__ Tok describe(const Args& a, const Row& r)
{
    Tok t{0, 0.0f, 0.0f, 0.0f, 0};
    if (!(r.flags & kFUsable))
        return t;
    if (!(r.flags & kFTest)) {
        t.ok = 1;
        return t;
    }
    const int x = __ldg(a.tok + (size_t)r.b * a.Kmax + r.i);
    bool ok = x >= 0 && x < a.V;
    if (!(r.flags & kFGreedy)) {
        t.u = __ldg(a.uni + (size_t)r.b * (a.Kmax + 1) + r.i);
        ok = ok && t.u >= 0.0f && t.u < 1.0f;
    }
    if (ok) {
        const size_t trow = (size_t)r.b * (a.Kmax + 1) + r.i;
        t.lt = Elem<T>::load(static_cast<const T*>(a.tgt) + trow * (size_t)a.V + x);
        if (r.flags & kFDraft)
            t.ld = Elem<T>::load(static_cast<const T*>(a.drf) +
                                 ((size_t)r.b * a.Kmax + r.i) * (size_t)a.V + x);
    }
    t.x = x;
    t.ok = ok ? 1 : 0;
    return t;
}

__device__ __forceinline__ Tok shfl_tok(const Tok& t)
{
    Tok o;
    o.x = __shfl_sync(kFull, t.x, 0);
    o.u = __shfl_sync(kFull, t.u, 0);
    o.lt = __shfl_sync(kFull, t.lt, 0);
    o.ld = __shfl_sync(kFull, t.ld, 0);
    o.ok = __shfl_sync(kFull, t.ok, 0);
    return o;
}

// Claim the next unit of work (one thread): a sequence id in claim order, or
// a live row index i * B + b when clusters claim single rows.  -1: none left.
// Anything outside the unit range also reads as -1, so a unit id can never
// index past the batch.
__device__ __forceinline__ int claim_unit(const Args& a)
{
    for (;;) {
        const int u = atomicAdd(a.next_unit, 1);
        if (u < 0 || u >= a.n_units)
            return -1;
        if (!a.per_row) {
            const int b = __ldg(a.order + u);
            return (b >= 0 && b < a.B) ? b : -1;
        }
        const int i = u / a.B;
        if (i <= __ldg(a.K + (u - i * a.B)))
            return u;
    }
}

__device__ __forceinline__ bool unit_valid(const Args& a, int u)
{
    return u >= 0 && u < (a.per_row ? a.n_units : a.B);
}

// First row of a claimed (valid) unit, with its sequence's K_b and T loaded
// but not yet used (the flags are made when the unit starts).
struct UnitPos {
    int i, b, Kb;
    float T;
};

__device__ __forceinline__ UnitPos unit_pos(const Args& a, int unit)
{
    UnitPos p;
    p.i = 0;
    p.b = unit;
    if (a.per_row) {
        p.i = unit / a.B;
        p.b = unit - p.i * a.B;
    }
    p.Kb = __ldg(a.K + p.b);
    p.T = __ldg(a.temp + p.b);
    return p;
}

__device__ __forceinline__ Row unit_row(const Args& a, int unit)
{
    const UnitPos p = unit_pos(a, unit);
    return make_row(a, p.i, p.b, p.Kb, p.T);
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
    // sum of exp2((l - m) c) over the lane's elements
    __device__ static __forceinline__ float exp_sum(const uint4 (&v)[NV], float m, float c)
    {
        const uint64_t M = f2_pack(m, m), Cc = f2_pack(c, c);
        uint64_t acc0 = f2_pack(0.0f, 0.0f), acc1 = acc0;
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const uint32_t wv[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                float d0, d1;
                f2_unpack(f2_mul(f2_sub(pair(wv[h]), M), Cc), d0, d1);
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
    // sums of the residual terms max(0, p - q) and of the weights of p
    __device__ static __forceinline__ void resid_sums(const uint4 (&t)[NV], const uint4 (&d)[NV],
                                                      float mt, float ist, float md, float isd,
                                                      float c, float& rs, float& ps)
    {
        const uint64_t MT = f2_pack(mt, mt), MD = f2_pack(md, md), Cc = f2_pack(c, c);
        const uint64_t IT = f2_pack(ist, ist), ID = f2_pack(isd, isd);
        uint64_t racc = f2_pack(0.0f, 0.0f), pacc = racc;
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const uint32_t wt[4] = {t[k].x, t[k].y, t[k].z, t[k].w};
            const uint32_t wd[4] = {d[k].x, d[k].y, d[k].z, d[k].w};
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                float a0, a1, b0, b1;
                f2_unpack(f2_mul(f2_sub(pair(wt[h]), MT), Cc), a0, a1);
                f2_unpack(f2_mul(f2_sub(pair(wd[h]), MD), Cc), b0, b1);
                const uint64_t et = f2_pack(ex2_approx(a0), ex2_approx(a1));
                const uint64_t ed = f2_pack(ex2_approx(b0), ex2_approx(b1));
                float r0, r1;
                f2_unpack(f2_sub(f2_mul(et, IT), f2_mul(ed, ID)), r0, r1);
                racc = f2_add(racc, f2_pack(fmaxf(r0, 0.0f), fmaxf(r1, 0.0f)));
                pacc = f2_add(pacc, et);
            }
        }
        float x0, x1, y0, y1;
        f2_unpack(racc, x0, x1);
        f2_unpack(pacc, y0, y1);
        rs = x0 + x1;
        ps = y0 + y1;
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
        const uint64_t M = f2_pack(m, m), Cc = f2_pack(c, c);
        uint64_t acc0 = f2_pack(0.0f, 0.0f), acc1 = acc0;
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            float d0, d1, d2, d3;
            f2_unpack(f2_mul(f2_sub(f2_pack(__uint_as_float(v[k].x), __uint_as_float(v[k].y)), M),
                             Cc), d0, d1);
            f2_unpack(f2_mul(f2_sub(f2_pack(__uint_as_float(v[k].z), __uint_as_float(v[k].w)), M),
                             Cc), d2, d3);
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
    __device__ static __forceinline__ void resid_sums(const uint4 (&t)[NV], const uint4 (&d)[NV],
                                                      float mt, float ist, float md, float isd,
                                                      float c, float& rs, float& ps)
    {
        const uint64_t MT = f2_pack(mt, mt), MD = f2_pack(md, md), Cc = f2_pack(c, c);
        const uint64_t IT = f2_pack(ist, ist), ID = f2_pack(isd, isd);
        uint64_t racc = f2_pack(0.0f, 0.0f), pacc = racc;
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const uint32_t wt[4] = {t[k].x, t[k].y, t[k].z, t[k].w};
            const uint32_t wd[4] = {d[k].x, d[k].y, d[k].z, d[k].w};
#pragma unroll
            for (int h = 0; h < 4; h += 2) {
                float a0, a1, b0, b1;
                f2_unpack(f2_mul(f2_sub(f2_pack(__uint_as_float(wt[h]), __uint_as_float(wt[h + 1])),
                                        MT), Cc), a0, a1);
                f2_unpack(f2_mul(f2_sub(f2_pack(__uint_as_float(wd[h]), __uint_as_float(wd[h + 1])),
                                        MD), Cc), b0, b1);
                const uint64_t et = f2_pack(ex2_approx(a0), ex2_approx(a1));
                const uint64_t ed = f2_pack(ex2_approx(b0), ex2_approx(b1));
                float r0, r1;
                f2_unpack(f2_sub(f2_mul(et, IT), f2_mul(ed, ID)), r0, r1);
                racc = f2_add(racc, f2_pack(fmaxf(r0, 0.0f), fmaxf(r1, 0.0f)));
                pacc = f2_add(pacc, et);
            }
        }
        float x0, x1, y0, y1;
        f2_unpack(racc, x0, x1);
        f2_unpack(pacc, y0, y1);
        rs = x0 + x1;
        ps = y0 + y1;
    }
};

// ---------------------------------------------------------------------------
// one warp's ring of stages
// ---------------------------------------------------------------------------
template <typename T, int NV>
struct Ring {
    static constexpr int CH = 32 * NV * Elem<T>::E;
    T* base;          // this warp's R stages
    uint64_t* bars;   // this warp's R mbarriers
    int R;
    __device__ T* tst(int s) const { return base + (size_t)s * 2 * CH; }
    __device__ T* dst(int s) const { return base + (size_t)s * 2 * CH + CH; }
    __device__ uint32_t bar(int s) const { return smem_addr(&bars[s]); }
};

// Copy number q (stage q % R) brings global chunk gc of a row: the
// 16-byte-aligned body by bulk copy, the ragged tail (or the whole chunk when
// rows are not 16-byte aligned) by element loads, -inf past V.  The stage's
// previous contents have been consumed by this warp (whole warp calls).
template <typename T, int NV>
__device__ __forceinline__ void issue_chunk(const Args& a, const Ring<T, NV>& rg, uint32_t q,
                                            int gc, const T* trow, const T* drow, bool load_d,
                                            int lane)
{
    using EL = Elem<T>;
    constexpr int CH = Ring<T, NV>::CH;
    const int s = (int)(q % (uint32_t)rg.R);
    const int e0 = gc * CH;
    const int n = min(CH, a.V - e0);
    const int nb = a.aligned ? ((n * (int)sizeof(T)) & ~15) / (int)sizeof(T) : 0;
    T* dt = rg.tst(s);
    T* dd = rg.dst(s);
    if (lane == 0) {
        const uint32_t bytes = (uint32_t)nb * (uint32_t)sizeof(T);
        const uint32_t tx = bytes * (load_d ? 2u : 1u);
        if (tx) {
            fence_proxy_async();
            mbar_arrive_expect_tx(rg.bar(s), tx);
            bulk_copy_g2s(smem_addr(dt), trow + e0, bytes, rg.bar(s));
            if (load_d)
                bulk_copy_g2s(smem_addr(dd), drow + e0, bytes, rg.bar(s));
        } else {
            mbar_arrive(rg.bar(s));
        }
    }
    for (int j = nb + lane; j < n; j += 32) {
        EL::copy(dt + j, trow + e0 + j);
        if (load_d)
            EL::copy(dd + j, drow + e0 + j);
    }
    for (int j = n + lane; j < CH; j += 32) {
        EL::set_neg_inf(dt + j);
        if (load_d)
            EL::set_neg_inf(dd + j);
    }
}

template <typename T, int NV>
__device__ __forceinline__ void load_stage(const T* p, int lane, uint4 (&v)[NV])
{
    const uint4* q = reinterpret_cast<const uint4*>(p);
#pragma unroll
    for (int k = 0; k < NV; ++k)
        v[k] = q[k * 32 + lane];
}

// Combine (max, sum relative to that max) parts held one per lane; the sum
// is compensated.  Every lane gets the same result.
__device__ __forceinline__ void combine_ms(float m_part, float s_part, float c, float& m, float& S)
{
    m = warp_max_nan(m_part);
    S = warp_sum_comp(m_part == -INFINITY ? 0.0f : s_part * weight(m_part, m, c));
}

template <typename T, int NV>
__global__ void __launch_bounds__(kMaxWarps * 32) sv_sweep_kernel(const Args a)
{
    using EL = Elem<T>;
    using LN = Lane<T, NV>;
    constexpr int E = EL::E;
    constexpr int CH = 32 * NV * E;
    extern __shared__ __align__(128) unsigned char dsm[];

    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int nw = (int)(blockDim.x >> 5);
    const int C = a.C, V = a.V, Kmax = a.Kmax, R = a.ring;
    const int P = C * nw;   // partials per row
    const uint32_t rank = cluster_ctarank();
    const int c0 = (int)rank * a.ncpc;
    const int nck = max(0, min(a.ncpc, a.nchunks - c0));
    const int kw = w < nck ? (nck - w + nw - 1) / nw : 0;   // chunks of this warp
    const bool resident = kw <= R;                          // residual pass needs no re-read
    const SweepLayout L = sweep_layout(nw, R, CH * (int)sizeof(T), a.kw);

    Ring<T, NV> rg;
    rg.base = reinterpret_cast<T*>(dsm) + (size_t)w * R * 2 * CH;
    rg.bars = reinterpret_cast<uint64_t*>(dsm + L.bars) + (size_t)w * R;
    rg.R = R;
    uint64_t* xbar = reinterpret_cast<uint64_t*>(dsm + L.xbar);
    float4* xbuf = reinterpret_cast<float4*>(dsm + L.xbuf);   // [2][kMaxParts]
    int* xclaim = reinterpret_cast<int*>(dsm + L.xclaim);     // [2]
    int* first = reinterpret_cast<int*>(dsm + L.first);       // [2]
    float2* stats = reinterpret_cast<float2*>(dsm + L.stats) + (size_t)w * a.kw;

    // ---- set-up: barriers, then the first unit from rank 0 (one per cluster:
    // taking a spare here as well would leave clusters idle when there are
    // fewer than twice as many units as clusters) ----
    if (lane == 0) {
        for (int s = 0; s < R; ++s)
            mbar_init(rg.bar(s), 1);
        if (w == 0) {
            mbar_init(smem_addr(&xbar[0]), 1);
            mbar_init(smem_addr(&xbar[1]), 1);
        }
        fence_mbar_init();
    }
    __syncthreads();
    cluster_arrive();   // every CTA's barriers exist before any peer signals them
    int f0 = -1;
    if (rank == 0 && w == 0) {
        if (lane == 0)
            f0 = claim_unit(a);
        f0 = __shfl_sync(kFull, f0, 0);
    }
    cluster_wait();
    if (rank == 0 && w == 0 && lane < C) {
        const uint32_t dst = map_to_rank(smem_addr(first), (uint32_t)lane);
        st_cluster_s32(dst, f0);
    }
    cluster_arrive();
    cluster_wait();

    // ---- per-warp schedule state (the same in every warp of the cluster) ----
    bool active = unit_valid(a, first[0]);
    int spare = -1;   // claimed during the first row
    UnitPos spare_pos{0, 0, 0, 0.0f};
    bool exhausted = false;
    bool triggered = false;
    bool broken = false;     // a stage wait gave up: no more copies, rows poisoned
    bool xbroken = false;    // an exchange wait gave up: leave the loop
    Row row = active ? unit_row(a, first[0]) : make_row(a, 0, 0, 0, 0.0f);
    Tok tk{0, 0.0f, 0.0f, 0.0f, 0};
    uint32_t qi = 0;   // copies issued by this warp
    uint32_t qw = 0;   // copies waited for by this warp
    // bound on the rows a cluster can process (guards the loop after a timeout)
    const long long max_rows = (long long)a.n_units * (Kmax + 1) + 2;

    const T* tgt = static_cast<const T*>(a.tgt);
    const T* drf = static_cast<const T*>(a.drf);
    auto row_ptrs = [&](const Row& r, const T*& tr, const T*& dr) {
        tr = tgt + ((size_t)r.b * (Kmax + 1) + r.i) * (size_t)V;
        dr = (r.flags & kFDraft) ? drf + ((size_t)r.b * Kmax + r.i) * (size_t)V : nullptr;
    };
    // first copies of a pass over a row (copy numbers qi, qi + 1, ...)
    auto prologue = [&](const Row& r, bool with_d) {
        const T* tr;
        const T* dr;
        row_ptrs(r, tr, dr);
        const int n = min(R, kw);
        for (int j = 0; j < n; ++j)
            issue_chunk<T, NV>(a, rg, qi + (uint32_t)j, c0 + w + j * nw, tr, dr, with_d, lane);
        qi += (uint32_t)n;
    };
    // wait for copy q (whole warp); false if any lane gave up (the copy then
    // stays outstanding for the wind-down)
    auto wait_copy = [&](uint32_t q) -> bool {
        const bool ok = mbar_wait_bounded(rg.bar((int)(q % (uint32_t)R)), (q / (uint32_t)R) & 1u,
                                          kWaitSpins);
        const bool all = !__any_sync(kFull, !ok);
        if (all)
            qw = q + 1;
        return all;
    };

    if (active) {
        if ((row.flags & kFUsable) && kw > 0)
            prologue(row, (row.flags & kFDraft) != 0);
        if (lane == 0)
            tk = describe<T>(a, row);
    }

    for (long long k = 0; active && k < max_rows; ++k) {
        if (exhausted && !triggered) {   // the finaliser may start launching
            griddep_launch_dependents();
            triggered = true;
        }
        const int p = (int)(k & 1);
        const uint32_t xpar = (uint32_t)((k >> 1) & 1);
        const bool greedy = (row.flags & kFGreedy) != 0;
        const bool test = (row.flags & kFTest) != 0;
        const bool draft = (row.flags & kFDraft) != 0;
        const bool usable = (row.flags & kFUsable) != 0;
        const bool load = usable && !broken && kw > 0;
        const float c = (usable && !greedy) ? log2e_over(row.T) : 0.0f;
        const bool want_claim = spare < 0 && !exhausted;
        if (w == 0 && lane == 0)
            mbar_arrive_expect_tx(smem_addr(&xbar[p]), (uint32_t)P * 16u + (want_claim ? 4u : 0u));
        int claimed = -1;
        if (rank == 0 && w == 0 && lane == 0 && want_claim)
            claimed = claim_unit(a);
        const T* tr;
        const T* dr;
        row_ptrs(row, tr, dr);

        // ---- one pass over this warp's chunks ----
        float4 part = make_float4(-INFINITY, 0.0f, -INFINITY, 0.0f);
        const uint32_t q0 = qi - (uint32_t)(load ? min(R, kw) : 0);   // this row's first copy
        if (greedy) {
            float gm = -INFINITY;
            int gi = INT_MAX;
            if (load) {
                for (int j = 0; j < kw; ++j) {
                    const uint32_t q = q0 + (uint32_t)j;
                    if (!broken && !wait_copy(q))
                        broken = true;
                    __syncwarp();
                    uint4 tv[NV];
                    load_stage<T, NV>(rg.tst((int)(q % (uint32_t)R)), lane, tv);
                    __syncwarp();
                    if (j + R < kw && !broken) {
                        issue_chunk<T, NV>(a, rg, qi, c0 + w + (j + R) * nw, tr, dr, false, lane);
                        ++qi;
                    }
                    const float cm = LN::max(tv);
                    if (cm > gm) {   // strictly greater: an earlier index keeps a tie
                        const int gbase = (c0 + w + j * nw) * CH;
                        int found = INT_MAX;
#pragma unroll
                        for (int e = NV * E - 1; e >= 0; --e)   // the lowest match wins
                            if (LN::elem(tv, e) == cm)
                                found = gbase + ((e / E) * 32 + lane) * E + (e % E);
                        gm = cm;
                        gi = found;
                    } else if (cm != cm) {
                        gm = cm;
                    }
                }
            }
            const float m = warp_max_nan(gm);
            const int gidx = __reduce_min_sync(kFull, gm == m ? gi : INT_MAX);
            part = make_float4(broken ? NAN : m, __int_as_float(gidx), -INFINITY, 0.0f);
        } else if (test) {
            float mt = -INFINITY, st = 0.0f, md = -INFINITY, sd = 0.0f;
            if (load) {
                for (int j = 0; j < kw; ++j) {
                    const uint32_t q = q0 + (uint32_t)j;
                    if (!broken && !wait_copy(q))
                        broken = true;
                    __syncwarp();
                    const int s = (int)(q % (uint32_t)R);
                    uint4 tv[NV], dv[NV];
                    load_stage<T, NV>(rg.tst(s), lane, tv);
                    if (draft)
                        load_stage<T, NV>(rg.dst(s), lane, dv);
                    __syncwarp();
                    if (j + R < kw && !broken) {
                        issue_chunk<T, NV>(a, rg, qi, c0 + w + (j + R) * nw, tr, dr, draft, lane);
                        ++qi;
                    }
                    const float nt = max_nan(mt, LN::max(tv));
                    if (nt != mt) {   // the lane max grew (or turned NaN): rescale the sum
                        st = mt == -INFINITY ? 0.0f : st * weight(mt, nt, c);
                        mt = nt;
                    }
                    st += LN::exp_sum(tv, mt == -INFINITY ? 0.0f : mt, c);
                    if (draft) {
                        const float nd = max_nan(md, LN::max(dv));
                        if (nd != md) {
                            sd = md == -INFINITY ? 0.0f : sd * weight(md, nd, c);
                            md = nd;
                        }
                        sd += LN::exp_sum(dv, md == -INFINITY ? 0.0f : md, c);
                    }
                }
            }
            float m1, S1, m2, S2;
            combine_ms(mt, st, c, m1, S1);
            combine_ms(md, sd, c, m2, S2);
            part = make_float4(broken ? NAN : m1, S1, m2, S2);
        } else {
            // bonus row: per-chunk (max, sum) of the target, kept for the draw
            if (load) {
                for (int j = 0; j < kw; ++j) {
                    const uint32_t q = q0 + (uint32_t)j;
                    if (!broken && !wait_copy(q))
                        broken = true;
                    __syncwarp();
                    uint4 tv[NV];
                    load_stage<T, NV>(rg.tst((int)(q % (uint32_t)R)), lane, tv);
                    __syncwarp();
                    if (j + R < kw && !broken) {
                        issue_chunk<T, NV>(a, rg, qi, c0 + w + (j + R) * nw, tr, dr, false, lane);
                        ++qi;
                    }
                    const float mc = warp_max_nan(LN::max(tv));
                    const float sc = mc == -INFINITY ? 0.0f : warp_sum(LN::exp_sum(tv, mc, c));
                    if (lane == 0)
                        stats[j] = make_float2(mc, sc);
                }
                __syncwarp();
            }
            // combine this warp's chunk stats, 32 at a time
            const int nst = load ? kw : 0;
            float mm = -INFINITY;
            for (int j = lane; j < nst; j += 32)
                mm = max_nan(mm, stats[j].x);
            const float mw = warp_max_nan(mm);
            float sacc = 0.0f, scmp = 0.0f;
            for (int j0 = 0; j0 < nst; j0 += 32) {
                const int j = j0 + lane;
                const float2 sj = j < nst ? stats[j] : make_float2(-INFINITY, 0.0f);
                const float v = warp_sum_comp(sj.x == -INFINITY ? 0.0f : sj.y * weight(sj.x, mw, c));
                float t, e;
                two_sum(sacc, v, t, e);
                sacc = t;
                scmp += e;
            }
            part = make_float4(broken ? NAN : mw, sacc + scmp, -INFINITY, 0.0f);
        }

        // ---- exchange: this warp's partial to every CTA of the cluster ----
        const int myslot = (int)rank * nw + w;
        const int claimed_b = __shfl_sync(kFull, claimed, 0);
        if (lane < C) {
            const uint32_t rb = map_to_rank(smem_addr(&xbar[p]), (uint32_t)lane);
            st_async_v4(map_to_rank(smem_addr(&xbuf[p * kMaxParts + myslot]), (uint32_t)lane), part,
                        rb);
            if (rank == 0 && w == 0 && want_claim)
                st_async_s32(map_to_rank(smem_addr(&xclaim[p]), (uint32_t)lane), claimed_b, rb);
        }
        if (!mbar_wait_bounded(smem_addr(&xbar[p]), xpar, kWaitSpins))
            xbroken = true;
        if (__any_sync(kFull, xbroken))
            break;

        // ---- combine all partials and decide (every warp alike) ----
        const float4 xv = lane < P ? xbuf[p * kMaxParts + lane]
                                   : make_float4(-INFINITY, __int_as_float(INT_MAX), -INFINITY, 0.0f);
        const Tok tkb = shfl_tok(tk);
        const size_t trow = (size_t)row.b * (Kmax + 1) + row.i;
        const bool writer = rank == 0 && w == 0 && lane == 0;
        int dec = kDecInvalid;
        float m_t = 0.0f, m_d = 0.0f, inv_st = 0.0f, inv_sd = 0.0f;
        bool row_ok = false;
        if (greedy) {
            m_t = warp_max_nan(xv.x);
            const int g =
                __reduce_min_sync(kFull, (lane < P && xv.x == m_t) ? __float_as_int(xv.y) : INT_MAX);
            row_ok = usable && tkb.ok && isfinite(m_t) && g < V;
            dec = !row_ok ? kDecInvalid : (test ? (tkb.x == g ? kDecAccept : kDecReject) : kDecBonus);
            if (writer) {
                a.dec[trow] = (uint8_t)dec;
                a.argmax[trow] = row_ok ? g : -1;
                if (test && a.want_pq) {
                    a.p_x[(size_t)row.b * Kmax + row.i] = NAN;
                    a.q_x[(size_t)row.b * Kmax + row.i] = NAN;
                }
            }
        } else {
            float St, Sd;
            combine_ms(xv.x, xv.y, c, m_t, St);
            combine_ms(xv.z, xv.w, c, m_d, Sd);
            row_ok = usable && tkb.ok && isfinite(m_t) && St > 0.0f &&
                     (!draft || (isfinite(m_d) && Sd > 0.0f));
            inv_st = row_ok ? __frcp_rn(St) : 0.0f;
            inv_sd = row_ok && draft ? __frcp_rn(Sd) : 0.0f;
            bool accept = false;
            float px = NAN, qx = NAN;
            if (test && row_ok) {
                px = __fmul_rn(weight(tkb.lt, m_t, c), inv_st);
                qx = __fmul_rn(weight(tkb.ld, m_d, c), inv_sd);
                accept = __fmul_rn(tkb.u, qx) < px;   // u < min(1, p/q) without a division
            }
            dec = !row_ok ? kDecInvalid : (test ? (accept ? kDecAccept : kDecReject) : kDecBonus);
            if (writer) {
                a.dec[trow] = (uint8_t)dec;
                a.rowstat[trow] = make_float4(m_t, inv_st, m_d, inv_sd);
                if (test && a.want_pq) {
                    a.p_x[(size_t)row.b * Kmax + row.i] = px;
                    a.q_x[(size_t)row.b * Kmax + row.i] = qx;
                }
            }
        }
        if (want_claim) {
            const int cl = xclaim[p];
            spare = unit_valid(a, cl) ? cl : -1;
            exhausted = spare < 0;
            if (spare >= 0)
                spare_pos = unit_pos(a, spare);   // loads now, used when the unit starts
        }

        // ---- chunk sums of p for the draw (bonus rows) ----
        if (!greedy && !test && row_ok && load) {
            for (int j = lane; j < kw; j += 32) {
                const float2 sj = stats[j];
                a.Pc[trow * a.nchunks + (c0 + w + j * nw)] =
                    sj.x == -INFINITY ? 0.0f : sj.y * weight(sj.x, m_t, c);
            }
        }
        // ---- residual pass: rows that may be drawn from ----
        if (!greedy && test && draft && row_ok && kw > 0 && !broken &&
            (dec == kDecReject || !a.early_exit)) {
            uint32_t r0 = q0;
            if (!resident) {
                r0 = qi;
                prologue(row, true);
            }
            for (int j = 0; j < kw; ++j) {
                const uint32_t q = r0 + (uint32_t)j;
                if (!resident) {
                    if (!broken && !wait_copy(q))
                        broken = true;
                    __syncwarp();
                }
                const int s = (int)(q % (uint32_t)R);
                uint4 tv[NV], dv[NV];
                load_stage<T, NV>(rg.tst(s), lane, tv);
                load_stage<T, NV>(rg.dst(s), lane, dv);
                __syncwarp();
                if (!resident && j + R < kw && !broken) {
                    issue_chunk<T, NV>(a, rg, qi, c0 + w + (j + R) * nw, tr, dr, true, lane);
                    ++qi;
                }
                float rs, ps;
                LN::resid_sums(tv, dv, m_t, inv_st, m_d, inv_sd, c, rs, ps);
                rs = warp_sum(rs);
                ps = warp_sum(ps);
                if (lane == 0) {
                    const size_t at = trow * a.nchunks + (c0 + w + j * nw);
                    a.Rc[at] = rs;
                    a.Pc[at] = ps;
                }
            }
        }

        // ---- the cluster's next row (the same decision in every warp) ----
        const bool valid = dec == kDecAccept || dec == kDecReject;
        const bool cont = !a.per_row && row.i < row.Kb &&
                          (dec == kDecAccept || (!a.early_exit && valid));
        if (cont) {
            row = make_row(a, row.i + 1, row.b, row.Kb, row.T);
        } else if (spare >= 0) {
            row = make_row(a, spare_pos.i, spare_pos.b, spare_pos.Kb, spare_pos.T);
            spare = -1;
        } else {
            break;
        }
        // copies first: the token loads of describe overlap with them
        if ((row.flags & kFUsable) && kw > 0 && !broken)
            prologue(row, (row.flags & kFDraft) != 0);
        if (lane == 0)
            tk = describe<T>(a, row);
    }

    // ---- wind-down: copies still in flight (only after a timeout), then
    // leave together, so that no CTA exits while a peer may still address it ----
    if (broken || xbroken) {
        if (lane == 0)
            atomicOr(a.err, kErrWaitTimeout);
        for (uint32_t q = qw; q < qi; ++q)
            (void)mbar_wait_bounded(rg.bar((int)(q % (uint32_t)R)), (q / (uint32_t)R) & 1u,
                                    kWaitSpins);
    }
    if (!triggered)
        griddep_launch_dependents();
    __syncwarp();
    cluster_arrive();
    cluster_wait();
}

}  // namespace sv
