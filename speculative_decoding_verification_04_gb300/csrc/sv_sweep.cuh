// sv_sweep.cuh -- the persistent vocabulary-sweep kernel.
//
// A grid of thread-block clusters (C CTAs each, as many as the device holds at
// once) works through the batch.  Each CTA owns `ncpc` contiguous vocabulary
// chunks of every row and keeps `nslot` shared-memory stages of that slice
// (target and draft), filled by 1-D bulk copies (cp.async.bulk, one mbarrier
// per chunk and stage).
//
// Schedule: every cluster runs `nslot` sequence slots round-robin, slot s
// using stage s.  A slot walks one sequence's positions in order.  As soon as
// row i is decided, the slot knows its next row exactly -- row i+1 when x_i was
// accepted, otherwise a fresh sequence (the rows after a rejection are never
// read: the method's own early exit, with no speculative traffic) -- and its
// bulk copies run while the cluster reduces the other slots' rows.  Fresh
// sequences come from one atomic claim per sequence (longest K first), made a
// whole row ahead by a scheduler warp.  When there are fewer sequences than
// clusters, slots claim single rows instead (all positions in parallel).
//
// Per row, with the slice resident in shared memory:
//   pass 1  per-warp NaN-propagating max of the target (and draft) logits;
//   pass 2  sampling rows: per-chunk sums of exp2((l - m_w) log2(e)/T) relative
//           to the warp max; greedy rows: lowest index of the warp max;
//   exchange  one cluster all-reduce through distributed shared memory of
//           (max, rescaled sum, argmax) per CTA;
//   decide  u q(x) < p(x) (sampling) or x == argmax (greedy);
//   pass 3  rejected rows (every tested row in verify-all mode): per-chunk
//           residual mass sum max(0, p - q) from the resident slice.
// Results go to the workspace; sv_finalize draws the tokens.
#pragma once

#include "sv_common.cuh"

namespace sv {

constexpr int kMaxSlots = 3;

// Row flags.  Schedule flags come from the sequence's K_b and T alone; the
// decision flag needs the proposed token and its uniform.
enum : int {
    kFGreedy = 1,   // T == 0
    kFTest = 2,     // i < K_b: a proposal is tested at this row
    kFDraft = 4,    // the draft row is read (tested sampling row)
    kFUsable = 8,   // temperature usable and, if needed, draft logits supplied
    kFOk = 16       // everything the decision needs is usable (set by describe)
};

// One row as every CTA of the cluster sees it (all fields derive from the
// same global reads, so every CTA takes the same branches).  Integer fields
// only: the struct lives in shared memory, shared by the CTA's threads.
struct Item {
    int i, b, Kb;
    float T;
    int sflags;         // kFGreedy | kFTest | kFDraft | kFUsable
    int x;
    float u;
    float lt_x, ld_x;   // target / draft logit at the proposed token (prefetched)
    int dflags;         // kFOk
};

// The row's schedule fields, from the sequence's cached K_b and T.
__device__ __forceinline__ Item schedule(const Args& a, int i, int b, int Kb, float T)
{
    Item it;
    it.i = i;
    it.b = b;
    it.Kb = Kb;
    it.T = T;
    const int greedy = T == 0.0f ? kFGreedy : 0;
    const int test = i < Kb ? kFTest : 0;
    const int draft = (test && !greedy) ? kFDraft : 0;
    const int usable = (temperature_usable(T) && (!draft || a.has_draft != 0)) ? kFUsable : 0;
    it.sflags = greedy | test | draft | usable;
    it.x = 0;
    it.u = it.lt_x = it.ld_x = 0.0f;
    it.dflags = 0;
    return it;
}

// Everything else the row's decision needs: the proposed token, its uniform
// and the two logits at the token (one thread; writes only x, u, lt_x, ld_x
// and dflags).  Called right after the row's bulk copies are issued, a full
// row ahead of the decision.
template <typename T>
__device__ __forceinline__ void describe(const Args& a, Item& it)
{
    const int f = it.sflags;
    if (!(f & kFUsable)) {
        it.dflags = 0;
        return;
    }
    if (!(f & kFTest)) {
        it.dflags = kFOk;
        return;
    }
    const int x = __ldg(a.tok + (size_t)it.b * a.Kmax + it.i);
    bool ok = x >= 0 && x < a.V;
    float u = 0.0f, lt = 0.0f, ld = 0.0f;
    if (!(f & kFGreedy)) {
        u = __ldg(a.uni + (size_t)it.b * (a.Kmax + 1) + it.i);
        ok = ok && u >= 0.0f && u < 1.0f;
    }
    if (ok) {
        const size_t trow = (size_t)it.b * (a.Kmax + 1) + it.i;
        lt = Elem<T>::load(static_cast<const T*>(a.tgt) + trow * (size_t)a.V + x);
        if ((f & kFDraft) && a.has_draft)
            ld = Elem<T>::load(static_cast<const T*>(a.drf) +
                               ((size_t)it.b * a.Kmax + it.i) * (size_t)a.V + x);
    }
    it.x = x;
    it.u = u;
    it.lt_x = lt;
    it.ld_x = ld;
    it.dflags = ok ? kFOk : 0;
}

// Claim the next unit of work (one thread): a sequence id in claim order, or
// a live row index i * B + b when slots claim single rows.  -1: none left.
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

// First row of a claimed unit.
__device__ __forceinline__ void unit_row(const Args& a, int unit, int* i, int* b)
{
    if (a.per_row) {
        *i = unit / a.B;
        *b = unit - *i * a.B;
    } else {
        *i = 0;
        *b = unit;
    }
}

template <typename T, int NV>
struct SweepSmem {
    static constexpr int E = Elem<T>::E;
    static constexpr int CH = 32 * NV * E;
    T* base;
    uint64_t* mbar;   // [nslot][ncpc]
    int ncpc;
    __device__ T* tchunk(int s, int lc) const { return base + ((size_t)s * 2 * ncpc + lc) * CH; }
    __device__ T* dchunk(int s, int lc) const { return base + ((size_t)s * 2 * ncpc + ncpc + lc) * CH; }
    __device__ uint32_t bar(int s, int lc) const { return smem_addr(&mbar[s * ncpc + lc]); }
};

// Stage this CTA's chunks of row `d` into stage `s` (compute warps only): the
// 16-byte-aligned body of each chunk by bulk copy, the ragged tail (or the
// whole chunk when rows are not 16-byte aligned) by element loads.  Every
// owned chunk's barrier receives exactly one arrival per use.
template <typename T, int NV>
__device__ __forceinline__ void issue_row(const Args& a, const SweepSmem<T, NV>& sm, const Item& d,
                                          int s, int c0, int nck, int cw, int nwc, int lane,
                                          bool poisoned)
{
    using EL = Elem<T>;
    constexpr int CH = SweepSmem<T, NV>::CH;
    const bool load_t = (d.sflags & kFUsable) && !poisoned;
    const bool load_d = load_t && (d.sflags & kFDraft) && a.has_draft != 0;
    const T* tg = static_cast<const T*>(a.tgt) + ((size_t)d.b * (a.Kmax + 1) + d.i) * (size_t)a.V;
    const T* dg = load_d ? static_cast<const T*>(a.drf) + ((size_t)d.b * a.Kmax + d.i) * (size_t)a.V
                         : nullptr;
    for (int lc = cw; lc < nck; lc += nwc) {
        const int e0 = (c0 + lc) * CH;
        const int n = min(CH, a.V - e0);
        const int nb = a.aligned ? ((n * (int)sizeof(T)) & ~15) / (int)sizeof(T) : 0;
        T* dt = sm.tchunk(s, lc);
        T* dd = sm.dchunk(s, lc);
        if (lane == 0) {
            const uint32_t mb = sm.bar(s, lc);
            const uint32_t bytes = (uint32_t)nb * (uint32_t)sizeof(T);
            const uint32_t tx = (load_t ? bytes : 0u) + (load_d ? bytes : 0u);
            if (tx) {
                fence_proxy_async();
                mbar_arrive_expect_tx(mb, tx);
                bulk_copy_g2s(smem_addr(dt), tg + e0, bytes, mb);
                if (load_d)
                    bulk_copy_g2s(smem_addr(dd), dg + e0, bytes, mb);
            } else {
                mbar_arrive(mb);
            }
        }
        if (load_t)
            for (int j = nb + lane; j < n; j += 32) {
                EL::copy(dt + j, tg + e0 + j);
                if (load_d)
                    EL::copy(dd + j, dg + e0 + j);
            }
    }
}

// A part's sum of exp2((l - m_part) c) rescaled to a common max m.  Parts
// whose max is -inf hold no mass.
__device__ __forceinline__ float rescaled(float s_part, float m_part, float m, float c)
{
    return m_part == -INFINITY ? 0.0f : s_part * weight(m_part, m, c);
}

// (max, sum, argmax) over up to 32 parts held one per lane, identical in every
// lane: NaN-propagating max, compensated sum of the rescaled part sums, lowest
// index among the parts holding the max.
__device__ __forceinline__ void combine_parts(float m_part, float s_part, int i_part, float c,
                                              float& m, float& S, int& idx)
{
    m = warp_max_nan(m_part);
    S = warp_sum_comp(rescaled(s_part, m_part, m, c));
    idx = __reduce_min_sync(kFull, m_part == m ? i_part : INT_MAX);
}

// Per-row result broadcast from warp 0 to the CTA.
struct RowResult {
    float m_t, m_d, inv_st, inv_sd;
    int dec;
    int resid;   // pass 3 wanted
};

// A sequence (or, in per-row mode, a row) held by a slot: the row it is at and
// the sequence's K_b and temperature, cached for its later rows.
struct SlotPos {
    int i, b, Kb;
    float T;
};

__device__ __forceinline__ SlotPos unit_pos(const Args& a, int unit)
{
    SlotPos p;
    unit_row(a, unit, &p.i, &p.b);
    p.Kb = __ldg(a.K + p.b);
    p.T = __ldg(a.temp + p.b);
    return p;
}

template <typename T, int NV>
__global__ void __launch_bounds__(kMaxWarps * 32, 1) sv_sweep_kernel(const Args a, const int nslot)
{
    using EL = Elem<T>;
    constexpr int E = EL::E;
    constexpr int CH = 32 * NV * E;

    extern __shared__ __align__(128) unsigned char dsmem[];
    __shared__ float s_wm[kMaxWarps][2];     // per compute warp: max (target, draft)
    __shared__ float s_ws[kMaxWarps][2];     // per compute warp: sum relative to its max
    __shared__ int s_wi[kMaxWarps];          // per compute warp: lowest index of its max
    // Exchange slots, double-buffered by row parity: a CTA can push row k+1's
    // partials while a peer still reads row k's; row k+2's push needs the row
    // k+1 barrier, which the peer reaches only after its reads.
    __shared__ float s_cm[2][kMaxCluster][2];   // per cluster rank, pushed: CTA max
    __shared__ float s_cs[2][kMaxCluster][2];   // per cluster rank, pushed: CTA sum
    __shared__ int s_ci[2][kMaxCluster];        // per cluster rank, pushed: CTA argmax
    __shared__ int s_claim[2];                  // unit claimed during the row, from rank 0
    __shared__ int s_units[kMaxSlots + 1];      // first units, pushed by rank 0
    __shared__ int s_bad;                       // a bounded copy wait gave up in this CTA
    __shared__ RowResult s_res;
    // Slot state, written by thread 0 (descriptors' decision fields by compute
    // warp 0, lane 0) between barriers and read by every thread.
    __shared__ Item s_desc[kMaxSlots];
    __shared__ int s_active[kMaxSlots];
    __shared__ int s_uses[kMaxSlots];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nwc = (int)(blockDim.x >> 5) - 1;   // compute warps; warp 0 schedules
    const int cw = warp - 1;                       // compute-warp index (-1: scheduler)
    const int C = a.C, V = a.V, Kmax = a.Kmax;
    const uint32_t rank = cluster_ctarank();
    const int c0 = (int)rank * a.ncpc;
    const int nck = max(0, min(a.ncpc, a.nchunks - c0));
    SweepSmem<T, NV> sm;
    sm.base = reinterpret_cast<T*>(dsmem);
    sm.ncpc = a.ncpc;
    sm.mbar = reinterpret_cast<uint64_t*>(dsmem + (size_t)nslot * 2 * a.ncpc * CH * sizeof(T));
    float* s_pc = reinterpret_cast<float*>(sm.mbar + (size_t)nslot * a.ncpc);   // [ncpc]

    // ---- one-time set-up: barriers, -inf padding past V (never overwritten) ----
    if (cw >= 0) {
        for (int lc = cw; lc < nck; lc += nwc) {
            if (lane == 0) {
                for (int s = 0; s < nslot; ++s)
                    mbar_init(sm.bar(s, lc), 1);
                fence_mbar_init();
            }
            const int n = min(CH, V - (c0 + lc) * CH);
            for (int s = 0; s < nslot; ++s)
                for (int j = n + lane; j < CH; j += 32) {
                    EL::set_neg_inf(sm.tchunk(s, lc) + j);
                    EL::set_neg_inf(sm.dchunk(s, lc) + j);
                }
        }
    }
    if (tid == 0)
        s_bad = 0;
    __syncthreads();

    // ---- first units: one per slot plus a spare (all CTAs started first) ----
    // The claims stay in warp 0's registers (lane 0 claims, a shuffle hands
    // them to the pushing lanes): nothing is read back from shared memory
    // that another thread wrote after its cluster arrive.
    cluster_arrive();
    int first[kMaxSlots + 1] = {-1, -1, -1, -1};
    if (rank == 0 && warp == 0) {
        if (lane == 0)
            for (int s = 0; s <= nslot; ++s)
                first[s] = claim_unit(a);
#pragma unroll
        for (int s = 0; s <= kMaxSlots; ++s)
            first[s] = __shfl_sync(kFull, first[s], 0);
    }
    cluster_wait();
    if (rank == 0 && tid < C) {
        const uint32_t dst = map_to_rank(smem_addr(&s_units[0]), (uint32_t)tid);
        for (int s = 0; s <= nslot; ++s)
            st_cluster_s32(dst + 4 * s, first[s]);
    }
    cluster_arrive();
    cluster_wait();

    // Slot state: the same in every CTA of the cluster (it derives from the
    // pushed units and from decisions every CTA computes identically).
    if (tid == 0) {
        for (int s = 0; s < kMaxSlots; ++s) {
            const int u = s < nslot ? s_units[s] : -1;
            s_uses[s] = 0;
            s_active[s] = unit_valid(a, u) ? 1 : 0;
            if (s_active[s]) {
                const SlotPos p = unit_pos(a, u);
                s_desc[s] = schedule(a, p.i, p.b, p.Kb, p.T);
            }
        }
    }
    __syncthreads();
    for (int s = 0; s < nslot; ++s) {
        if (!s_active[s])
            continue;
        if (cw >= 0)
            issue_row<T, NV>(a, sm, s_desc[s], s, c0, nck, cw, nwc, lane, false);
        if (cw == 0 && lane == 0)
            describe<T>(a, s_desc[s]);
    }
    __syncthreads();
    int spare = unit_valid(a, s_units[nslot]) ? s_units[nslot] : -1;
    SlotPos spare_pos{0, 0, 0, 0.0f};
    if (spare >= 0)
        spare_pos = unit_pos(a, spare);
    bool exhausted = spare < 0;
    bool triggered = false;
    int xp = 0;   // exchange parity: flips once per processed row

    for (int k = 0;; ++k) {
        const bool any = (s_active[0] | s_active[1] | s_active[2]) != 0;
        if (!any)
            break;
        if (exhausted && !triggered) {   // the finaliser may start launching
            griddep_launch_dependents();
            triggered = true;
        }
        const int s = k % nslot;
        if (!s_active[s])
            continue;
        const Item dc = s_desc[s];
        const bool d_greedy = (dc.sflags & kFGreedy) != 0;
        const bool d_test = (dc.sflags & kFTest) != 0;
        const bool d_draft = (dc.sflags & kFDraft) != 0;
        const bool d_ok = (dc.sflags & kFUsable) && (dc.dflags & kFOk);
        const uint32_t par = (uint32_t)s_uses[s] & 1u;
        const bool want_claim = spare < 0 && !exhausted;
        const bool poisoned_before = s_bad != 0;
        const float c = (d_ok && !d_greedy) ? log2e_over(dc.T) : 0.0f;
        const size_t trow = (size_t)dc.b * (Kmax + 1) + dc.i;

        float wmt = -INFINITY;   // this warp's target max (kept for its chunk sums)
        if (warp == 0) {
            // ---- scheduler: claim the next unit concurrently with the passes ----
            if (rank == 0 && lane == 0 && want_claim)
                s_claim[xp] = claim_unit(a);
        } else {
            // ---- pass 1: per-warp maxima over the owned chunks ----
            float mt[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
            float md[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
            bool timed = false;
            for (int lc = cw; lc < nck; lc += nwc) {
                if (!poisoned_before && !mbar_wait_bounded(sm.bar(s, lc), par, kWaitSpins))
                    timed = true;
                if (!d_ok)
                    continue;
                const uint4* vt = reinterpret_cast<const uint4*>(sm.tchunk(s, lc));
#pragma unroll
                for (int v = 0; v < NV; ++v) {
                    float xs[E];
                    EL::unpack(vt[v * 32 + lane], xs);
#pragma unroll
                    for (int e = 0; e < E; ++e)
                        mt[e & 3] = max_nan(mt[e & 3], xs[e]);
                }
                if (d_draft) {
                    const uint4* vd = reinterpret_cast<const uint4*>(sm.dchunk(s, lc));
#pragma unroll
                    for (int v = 0; v < NV; ++v) {
                        float xs[E];
                        EL::unpack(vd[v * 32 + lane], xs);
#pragma unroll
                        for (int e = 0; e < E; ++e)
                            md[e & 3] = max_nan(md[e & 3], xs[e]);
                    }
                }
            }
            if (__any_sync(kFull, timed) && lane == 0)
                s_bad = 1;
            wmt = warp_max_nan(max_nan(max_nan(mt[0], mt[1]), max_nan(mt[2], mt[3])));
            const float wmd = warp_max_nan(max_nan(max_nan(md[0], md[1]), max_nan(md[2], md[3])));
            int widx = INT_MAX;
            float wst = 0.0f, wsd = 0.0f;
            if (d_ok && d_greedy) {
                // ---- pass 2 (greedy): lowest index holding this warp's max ----
                if (isfinite(wmt)) {
                    for (int lc = cw; lc < nck; lc += nwc) {
                        const uint4* vt = reinterpret_cast<const uint4*>(sm.tchunk(s, lc));
                        const int gbase = (c0 + lc) * CH;
#pragma unroll
                        for (int v = 0; v < NV; ++v) {
                            float xs[E];
                            EL::unpack(vt[v * 32 + lane], xs);
#pragma unroll
                            for (int e = 0; e < E; ++e)
                                if (xs[e] == wmt)
                                    widx = min(widx, gbase + (v * 32 + lane) * E + e);
                        }
                    }
                }
                widx = __reduce_min_sync(kFull, widx);
            } else if (d_ok) {
                // ---- pass 2 (sampling): per-chunk sums relative to this warp's max ----
                for (int lc = cw; lc < nck; lc += nwc) {
                    float pc = 0.0f;
                    if (wmt != -INFINITY) {
                        const uint4* vt = reinterpret_cast<const uint4*>(sm.tchunk(s, lc));
                        float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
                        for (int v = 0; v < NV; ++v) {
                            float xs[E];
                            EL::unpack(vt[v * 32 + lane], xs);
#pragma unroll
                            for (int e = 0; e < E; ++e)
                                acc[e & 3] += weight(xs[e], wmt, c);
                        }
                        pc = warp_sum((acc[0] + acc[1]) + (acc[2] + acc[3]));
                    }
                    if (lane == 0)
                        s_pc[lc] = pc;
                    wst += pc;
                    if (d_draft && wmd != -INFINITY) {
                        const uint4* vd = reinterpret_cast<const uint4*>(sm.dchunk(s, lc));
                        float accd[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
                        for (int v = 0; v < NV; ++v) {
                            float xs[E];
                            EL::unpack(vd[v * 32 + lane], xs);
#pragma unroll
                            for (int e = 0; e < E; ++e)
                                accd[e & 3] += weight(xs[e], wmd, c);
                        }
                        wsd += warp_sum((accd[0] + accd[1]) + (accd[2] + accd[3]));
                    }
                }
            }
            if (lane == 0) {
                s_wm[cw][0] = wmt;
                s_wm[cw][1] = wmd;
                s_ws[cw][0] = wst;
                s_ws[cw][1] = wsd;
                s_wi[cw] = widx;
            }
        }
        __syncthreads();
        // ---- warp 0: this CTA's partial (lane w = compute warp w), pushed to every rank ----
        if (warp == 0) {
            const bool has = lane < nwc;
            float m0, m1, S0, S1;
            int i0, i1;
            combine_parts(has ? s_wm[lane][0] : -INFINITY, has ? s_ws[lane][0] : 0.0f,
                          has ? s_wi[lane] : INT_MAX, c, m0, S0, i0);
            combine_parts(has ? s_wm[lane][1] : -INFINITY, has ? s_ws[lane][1] : 0.0f, INT_MAX, c,
                          m1, S1, i1);
            if (s_bad) {   // poison this row in every CTA of the cluster
                m0 = NAN;
                m1 = NAN;
            }
            if (lane < C) {
                const uint32_t dm = map_to_rank(smem_addr(&s_cm[xp][rank][0]), (uint32_t)lane);
                st_cluster_f32(dm, m0);
                st_cluster_f32(dm + 4, m1);
                const uint32_t ds = map_to_rank(smem_addr(&s_cs[xp][rank][0]), (uint32_t)lane);
                st_cluster_f32(ds, S0);
                st_cluster_f32(ds + 4, S1);
                st_cluster_s32(map_to_rank(smem_addr(&s_ci[xp][rank]), (uint32_t)lane), i0);
                if (rank == 0 && want_claim) {
                    const int cl = s_claim[xp];
                    st_cluster_s32(map_to_rank(smem_addr(&s_claim[xp]), (uint32_t)lane), cl);
                }
                fence_cluster();   // the pushes above are released to the peers
            }
        }
        cluster_arrive_relaxed();
        cluster_wait();   // the one cluster exchange of this row (acquire)

        // ---- warp 0: cluster combine (lane r = rank r) and the decision ----
        if (warp == 0) {
            const bool has = lane < C;
            float m_t, m_d, St, Sd;
            int g, unused;
            combine_parts(has ? s_cm[xp][lane][0] : -INFINITY, has ? s_cs[xp][lane][0] : 0.0f,
                          has ? s_ci[xp][lane] : INT_MAX, c, m_t, St, g);
            combine_parts(has ? s_cm[xp][lane][1] : -INFINITY, has ? s_cs[xp][lane][1] : 0.0f,
                          INT_MAX, c, m_d, Sd, unused);
            if (lane == 0) {
                const bool ok_t = isfinite(m_t);
                const bool ok_d = !d_draft || isfinite(m_d);
                RowResult res{m_t, m_d, 0.0f, 0.0f, kDecInvalid, 0};
                if (d_greedy) {
                    const bool row_ok = d_ok && ok_t && g < V;
                    res.dec = !row_ok ? kDecInvalid
                                      : (d_test ? (dc.x == g ? kDecAccept : kDecReject)
                                                    : kDecBonus);
                    if (rank == 0) {
                        a.dec[trow] = (uint8_t)res.dec;
                        a.argmax[trow] = row_ok ? g : -1;
                        if (d_test && a.want_pq) {
                            a.p_x[(size_t)dc.b * Kmax + dc.i] = NAN;
                            a.q_x[(size_t)dc.b * Kmax + dc.i] = NAN;
                        }
                    }
                } else {
                    const bool row_ok =
                        d_ok && ok_t && ok_d && St > 0.0f && (!d_draft || Sd > 0.0f);
                    res.inv_st = row_ok ? __frcp_rn(St) : 0.0f;
                    res.inv_sd = row_ok && d_draft ? __frcp_rn(Sd) : 0.0f;
                    bool accept = false;
                    float px = NAN, qx = NAN;
                    if (d_test && row_ok) {
                        px = __fmul_rn(weight(dc.lt_x, m_t, c), res.inv_st);
                        qx = __fmul_rn(weight(dc.ld_x, m_d, c), res.inv_sd);
                        accept = __fmul_rn(dc.u, qx) < px;   // u < min(1, p/q) without a division
                    }
                    res.dec = !row_ok ? kDecInvalid
                                      : (d_test ? (accept ? kDecAccept : kDecReject) : kDecBonus);
                    res.resid = row_ok && d_draft && (res.dec == kDecReject || !a.early_exit);
                    if (rank == 0) {
                        a.dec[trow] = (uint8_t)res.dec;
                        a.rowstat[trow] = make_float4(m_t, res.inv_st, m_d, res.inv_sd);
                        if (d_test && a.want_pq) {
                            a.p_x[(size_t)dc.b * Kmax + dc.i] = px;
                            a.q_x[(size_t)dc.b * Kmax + dc.i] = qx;
                        }
                    }
                }
                s_res = res;
            }
        }
        __syncthreads();
        const RowResult res = s_res;

        // ---- next row of this slot (same decision in every thread), issued at once ----
        if (want_claim) {
            spare = unit_valid(a, s_claim[xp]) ? s_claim[xp] : -1;
            exhausted = spare < 0;
            if (spare >= 0)
                spare_pos = unit_pos(a, spare);
        }
        xp ^= 1;
        const bool valid = res.dec == kDecAccept || res.dec == kDecReject;
        const bool cont = !a.per_row && dc.i < dc.Kb &&
                          (res.dec == kDecAccept || (!a.early_exit && valid));
        SlotPos np{dc.i + 1, dc.b, dc.Kb, dc.T};
        bool next_active = true;
        if (!cont) {
            if (spare >= 0) {
                np = spare_pos;
                spare = -1;
            } else {
                next_active = false;
            }
        }

        if (cw >= 0 && !d_greedy && res.dec != kDecInvalid) {
            // chunk sums of the weights, rescaled to the row max
            if (lane == 0)
                for (int lc = cw; lc < nck; lc += nwc)
                    a.Pc[trow * a.nchunks + (c0 + lc)] =
                        wmt == -INFINITY ? 0.0f : s_pc[lc] * weight(wmt, res.m_t, c);
            // ---- pass 3: residual mass per chunk of rows that may be drawn from ----
            if (res.resid) {
                for (int lc = cw; lc < nck; lc += nwc) {
                    const uint4* vt = reinterpret_cast<const uint4*>(sm.tchunk(s, lc));
                    const uint4* vd = reinterpret_cast<const uint4*>(sm.dchunk(s, lc));
                    float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
                    for (int v = 0; v < NV; ++v) {
                        float xt[E], xd[E];
                        EL::unpack(vt[v * 32 + lane], xt);
                        EL::unpack(vd[v * 32 + lane], xd);
#pragma unroll
                        for (int e = 0; e < E; ++e)
                            acc[e & 3] += resid_term(weight(xt[e], res.m_t, c), res.inv_st,
                                                     weight(xd[e], res.m_d, c), res.inv_sd);
                    }
                    const float rc = warp_sum((acc[0] + acc[1]) + (acc[2] + acc[3]));
                    if (lane == 0)
                        a.Rc[trow * a.nchunks + (c0 + lc)] = rc;
                }
            }
        }
        if (tid == 0) {
            if (s_bad && !poisoned_before)
                atomicOr(a.err, kErrWaitTimeout);
            // nobody reads slot s's shared state again before the barrier below
            s_uses[s] += 1;
            s_active[s] = next_active ? 1 : 0;
            if (next_active)
                s_desc[s] = schedule(a, np.i, np.b, np.Kb, np.T);
        }
        __syncthreads();   // stage s consumed; s_pc, s_w*, s_res free; slot s rescheduled
        if (next_active) {
            if (cw >= 0)
                issue_row<T, NV>(a, sm, s_desc[s], s, c0, nck, cw, nwc, lane, s_bad != 0);
            if (cw == 0 && lane == 0)
                describe<T>(a, s_desc[s]);
        }
        // If the next row processed is this slot's again (one slot, or the
        // other slots idle), its descriptor must be complete before it is read.
        bool same_next = true;
        for (int t = 1; t < nslot; ++t)
            if (s_active[(s + t) % nslot]) {
                same_next = false;
                break;
            }
        if (same_next)
            __syncthreads();
    }
}

}  // namespace sv
