// sv_sweep.cuh -- the persistent vocabulary-sweep kernel.
//
// A grid of thread-block clusters (C CTAs each, one cluster per GPC slot the
// device can hold) loops over the (position i, sequence b) rows of the batch in
// position-major order.  Each CTA owns `ncpc` contiguous vocabulary chunks of
// every row; its shared memory holds `stages` copies of that slice (target and
// draft), filled by 1-D bulk copies (cp.async.bulk, one mbarrier per chunk and
// stage).  With two stages the copies of row k+1 land while row k is reduced.
//
// Per row, with the slice resident in shared memory:
//   pass 1  NaN-propagating max of the target (and draft) logits, warp
//           shuffles, cluster all-reduce through distributed shared memory;
//   pass 2  sampling rows: per-chunk sums of exp2((l - m) log2(e)/T) for
//           target and draft, cluster all-reduce of S_t, S_d;
//           greedy rows: lowest index holding the maximum;
//   decide  u q(x) < p(x) (sampling) or x == argmax (greedy), identically in
//           every CTA; a rejection or unusable row sets the sequence's mask bit
//           so that later positions of the sequence are never claimed;
//   pass 3  rejected rows (every tested row in verify-all mode): per-chunk
//           residual mass sum max(0, p - q).
// Results go to the workspace; sv_finalize draws the tokens.
#pragma once

#include "sv_common.cuh"

namespace sv {

// One row as every CTA of the cluster sees it (all fields derive from the
// same global reads, so every CTA takes the same branches).
struct Item {
    int idx;   // position-major row index, -1 = none
    int i, b, Kb;
    float T;
    int x;
    float u;
    bool ok;   // temperature, token, uniform and draft pointer usable
    bool greedy, is_test, use_draft;
};

__device__ __forceinline__ Item describe(const Args& a, int idx)
{
    Item it;
    it.idx = idx;
    it.i = it.b = it.Kb = it.x = 0;
    it.T = it.u = 0.0f;
    it.ok = it.greedy = it.is_test = it.use_draft = false;
    if (idx < 0)
        return it;
    it.i = idx / a.B;
    it.b = idx - it.i * a.B;
    it.Kb = __ldg(a.K + it.b);
    it.T = __ldg(a.temp + it.b);
    it.greedy = it.T == 0.0f;
    it.is_test = it.i < it.Kb;
    it.use_draft = it.is_test && !it.greedy;
    bool ok = temperature_usable(it.T);
    if (it.is_test) {
        it.x = __ldg(a.tok + (size_t)it.b * a.Kmax + it.i);
        ok = ok && it.x >= 0 && it.x < a.V;
        if (!it.greedy) {
            it.u = __ldg(a.uni + (size_t)it.b * (a.Kmax + 1) + it.i);
            ok = ok && it.u >= 0.0f && it.u < 1.0f && a.drf != nullptr;
        }
    }
    it.ok = ok;
    return it;
}

// A known earlier rejection (or unusable row) of sequence b makes position i moot.
__device__ __forceinline__ bool row_moot(const Args& a, int i, int b)
{
    if (!a.early_exit || i == 0)
        return false;
    return (ld_volatile_u32(a.mask + b) & positions_below(i)) != 0;
}

// Claimed-but-unprocessed rows of one cluster, held by warp 0 of rank 0:
// lane j keeps the j-th queued row index in qv.
struct ClaimQueue {
    int qv, qn, qh, qw;
};

// Warp-cooperative claim of the next row that needs work.  All 32 lanes call
// it and get the same result.  Padding rows (i > K_b) and rows made moot by
// an earlier rejection are dropped here, so they cost the cluster no barrier;
// the claim width adapts to how many claimed rows turn out to be needed.
__device__ int claim_row(const Args& a, ClaimQueue& q, int lane)
{
    for (;;) {
        while (q.qh < q.qn) {
            const int idx = __shfl_sync(kFull, q.qv, q.qh);
            ++q.qh;
            int moot = 0;
            if (lane == 0) {
                const int i = idx / a.B;
                moot = row_moot(a, i, idx - i * a.B);
            }
            if (!__shfl_sync(kFull, moot, 0))
                return idx;
        }
        int base = 0;
        if (lane == 0)
            base = atomicAdd(a.next_item, q.qw);
        base = __shfl_sync(kFull, base, 0);
        if (base >= a.n_items) {
            q.qn = q.qh = 0;
            return -1;
        }
        const int idx = base + lane;
        bool need = false;
        if (lane < q.qw && idx < a.n_items) {
            const int i = idx / a.B, b = idx - i * a.B;
            need = i <= __ldg(a.K + b) && !row_moot(a, i, b);
        }
        const unsigned bal = __ballot_sync(kFull, need);
        const int cnt = __popc(bal);
        const int src = lane < cnt ? (int)__fns(bal, 0, lane + 1) : 0;
        q.qv = __shfl_sync(kFull, idx, src);
        q.qn = cnt;
        q.qh = 0;
        q.qw = cnt == 0 ? min(32, 2 * q.qw) : (cnt >= 2 ? max(1, q.qw / 2) : q.qw);
    }
}

template <typename T, int NV>
struct SweepSmem {
    static constexpr int E = Elem<T>::E;
    static constexpr int CH = 32 * NV * E;
    T* base;
    uint64_t* mbar;   // [stages][ncpc]
    int ncpc;
    __device__ T* tchunk(int s, int lc) const { return base + ((size_t)s * 2 * ncpc + lc) * CH; }
    __device__ T* dchunk(int s, int lc) const { return base + ((size_t)s * 2 * ncpc + ncpc + lc) * CH; }
    __device__ uint32_t bar(int s, int lc) const { return smem_addr(&mbar[s * ncpc + lc]); }
};

// Stage this CTA's chunks of row `d` into stage `s`: the 16-byte-aligned body
// of each chunk by bulk copy, the ragged tail (or the whole chunk when rows
// are not 16-byte aligned) by element loads.  Every owned chunk's barrier
// receives exactly one arrival per use, whether or not anything is copied.
template <typename T, int NV>
__device__ __forceinline__ void issue_row(const Args& a, const SweepSmem<T, NV>& sm, const Item& d,
                                          int s, int c0, int nck, int warp, int nw, int lane,
                                          bool poisoned)
{
    using EL = Elem<T>;
    constexpr int CH = SweepSmem<T, NV>::CH;
    const bool load_t = d.ok && !poisoned;
    const bool load_d = load_t && d.use_draft;
    const T* tg = static_cast<const T*>(a.tgt) + ((size_t)d.b * (a.Kmax + 1) + d.i) * (size_t)a.V;
    const T* dg = load_d ? static_cast<const T*>(a.drf) + ((size_t)d.b * a.Kmax + d.i) * (size_t)a.V
                         : nullptr;
    for (int lc = warp; lc < nck; lc += nw) {
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

template <typename T, int NV>
__global__ void __launch_bounds__(kMaxWarps * 32, 1) sv_sweep_kernel(const Args a, const int stages)
{
    using EL = Elem<T>;
    constexpr int E = EL::E;
    constexpr int CH = 32 * NV * E;

    extern __shared__ __align__(128) unsigned char dsmem[];
    __shared__ float s_wmax[kMaxWarps][2];
    __shared__ double s_wsum[kMaxWarps][2];
    __shared__ int s_widx[kMaxWarps];
    __shared__ float s_cmax[kMaxCluster][2];    // one slot per cluster rank
    __shared__ double s_csum[kMaxCluster][2];
    __shared__ int s_cidx[kMaxCluster];
    __shared__ int s_first[2];                  // first two rows, pushed by rank 0
    __shared__ int s_next;                      // row after next, pushed by rank 0
    __shared__ int s_bad;                       // a bounded copy wait gave up in this CTA

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
    const int C = a.C, V = a.V, Kmax = a.Kmax;
    const uint32_t rank = cluster_ctarank();
    const int c0 = (int)rank * a.ncpc;
    const int nck = max(0, min(a.ncpc, a.nchunks - c0));
    SweepSmem<T, NV> sm;
    sm.base = reinterpret_cast<T*>(dsmem);
    sm.ncpc = a.ncpc;
    sm.mbar = reinterpret_cast<uint64_t*>(dsmem + (size_t)stages * 2 * a.ncpc * CH * sizeof(T));

    // ---- one-time set-up: barriers, -inf padding past V (never overwritten) ----
    for (int lc = warp; lc < nck; lc += nw) {
        if (lane == 0) {
            for (int s = 0; s < stages; ++s)
                mbar_init(sm.bar(s, lc), 1);
            fence_mbar_init();
        }
        const int n = min(CH, V - (c0 + lc) * CH);
        for (int s = 0; s < stages; ++s)
            for (int j = n + lane; j < CH; j += 32) {
                EL::set_neg_inf(sm.tchunk(s, lc) + j);
                EL::set_neg_inf(sm.dchunk(s, lc) + j);
            }
    }
    if (tid == 0)
        s_bad = 0;
    __syncthreads();

    // ---- first two rows (all CTAs started before any DSMEM store) ----
    ClaimQueue q{0, 0, 0, 1};
    cluster_arrive();
    int r0 = -1, r1 = -1;
    if (rank == 0 && warp == 0) {
        r0 = claim_row(a, q, lane);
        r1 = r0 >= 0 ? claim_row(a, q, lane) : -1;
    }
    cluster_wait();
    if (rank == 0 && tid < C) {
        const uint32_t dst = map_to_rank(smem_addr(&s_first[0]), (uint32_t)tid);
        st_cluster_s32(dst, r0);
        st_cluster_s32(dst + 4, r1);
    }
    cluster_arrive();
    cluster_wait();

    Item dc = describe(a, s_first[0]);
    Item dn = describe(a, s_first[1]);
    if (dc.idx >= 0)
        issue_row<T, NV>(a, sm, dc, 0, c0, nck, warp, nw, lane, false);
    bool triggered = false;

    for (int k = 0; dc.idx >= 0; ++k) {
        const int st = k % stages;
        const uint32_t par = (uint32_t)(k / stages) & 1u;
        if (stages == 2 && dn.idx >= 0)
            issue_row<T, NV>(a, sm, dn, st ^ 1, c0, nck, warp, nw, lane, s_bad != 0);
        if (dn.idx < 0 && !triggered) {
            griddep_launch_dependents();
            triggered = true;
        }
        int nn = -1;
        if (rank == 0 && warp == 0)
            nn = claim_row(a, q, lane);

        const bool poisoned_before = s_bad != 0;
        // ---- pass 1: maxima ----
        float mt[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
        float md[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
        bool timed = false;
        for (int lc = warp; lc < nck; lc += nw) {
            if (!poisoned_before && !mbar_wait_bounded(sm.bar(st, lc), par, kWaitSpins))
                timed = true;
            if (!dc.ok)
                continue;
            const uint4* vt = reinterpret_cast<const uint4*>(sm.tchunk(st, lc));
#pragma unroll
            for (int v = 0; v < NV; ++v) {
                float xs[E];
                EL::unpack(vt[v * 32 + lane], xs);
#pragma unroll
                for (int e = 0; e < E; ++e)
                    mt[e & 3] = max_nan(mt[e & 3], xs[e]);
            }
            if (dc.use_draft) {
                const uint4* vd = reinterpret_cast<const uint4*>(sm.dchunk(st, lc));
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
        float wmt = warp_max_nan(max_nan(max_nan(mt[0], mt[1]), max_nan(mt[2], mt[3])));
        float wmd = warp_max_nan(max_nan(max_nan(md[0], md[1]), max_nan(md[2], md[3])));
        if (lane == 0) {
            s_wmax[warp][0] = wmt;
            s_wmax[warp][1] = wmd;
        }
        __syncthreads();
        if (tid < C) {
            float cm0 = -INFINITY, cm1 = -INFINITY;
            for (int w = 0; w < nw; ++w) {
                cm0 = max_nan(cm0, s_wmax[w][0]);
                cm1 = max_nan(cm1, s_wmax[w][1]);
            }
            if (s_bad) {   // poison this row in every CTA of the cluster
                cm0 = NAN;
                cm1 = NAN;
            }
            const uint32_t dst = map_to_rank(smem_addr(&s_cmax[rank][0]), (uint32_t)tid);
            st_cluster_f32(dst, cm0);
            st_cluster_f32(dst + 4, cm1);
            if (rank == 0)
                st_cluster_s32(map_to_rank(smem_addr(&s_next), (uint32_t)tid), nn);
        }
        cluster_arrive();
        cluster_wait();   // B
        const Item dnn = describe(a, s_next);
        float m_t = -INFINITY, m_d = -INFINITY;
        for (int r = 0; r < C; ++r) {
            m_t = max_nan(m_t, s_cmax[r][0]);
            m_d = max_nan(m_d, s_cmax[r][1]);
        }
        const bool ok_t = isfinite(m_t);
        const bool ok_d = !dc.use_draft || isfinite(m_d);
        const size_t trow = (size_t)dc.b * (Kmax + 1) + dc.i;
        const bool work = dc.ok && ok_t && ok_d;

        if (dc.greedy) {
            // ---- pass 2 (greedy): lowest index holding the max ----
            int best = INT_MAX;
            if (work) {
                for (int lc = warp; lc < nck; lc += nw) {
                    const uint4* vt = reinterpret_cast<const uint4*>(sm.tchunk(st, lc));
                    const int gbase = (c0 + lc) * CH;
#pragma unroll
                    for (int v = 0; v < NV; ++v) {
                        float xs[E];
                        EL::unpack(vt[v * 32 + lane], xs);
#pragma unroll
                        for (int e = 0; e < E; ++e)
                            if (xs[e] == m_t)
                                best = min(best, gbase + (v * 32 + lane) * E + e);
                    }
                }
            }
            best = __reduce_min_sync(kFull, best);
            if (lane == 0)
                s_widx[warp] = best;
            __syncthreads();
            if (tid < C) {
                int cb = INT_MAX;
                for (int w = 0; w < nw; ++w)
                    cb = min(cb, s_widx[w]);
                st_cluster_s32(map_to_rank(smem_addr(&s_cidx[rank]), (uint32_t)tid), cb);
            }
            cluster_arrive();
            cluster_wait();   // C
            int g = INT_MAX;
            for (int r = 0; r < C; ++r)
                g = min(g, s_cidx[r]);
            const bool row_ok = work && g < V;
            const uint8_t d = !row_ok ? kDecInvalid
                                      : (dc.is_test ? (dc.x == g ? kDecAccept : kDecReject) : kDecBonus);
            if (rank == 0 && tid == 0) {
                if (dc.is_test && d != kDecAccept)
                    atomicOr(a.mask + dc.b, 1u << dc.i);
                a.dec[trow] = d;
                a.argmax[trow] = row_ok ? g : -1;
                if (dc.is_test && a.p_x) {
                    a.p_x[(size_t)dc.b * Kmax + dc.i] = NAN;
                    a.q_x[(size_t)dc.b * Kmax + dc.i] = NAN;
                }
            }
        } else {
            // ---- pass 2 (sampling): per-chunk sums of the softmax weights ----
            const float c = dc.ok ? (float)(kLog2e / (double)dc.T) : 0.0f;
            double wst = 0.0, wsd = 0.0;
            if (work) {
                for (int lc = warp; lc < nck; lc += nw) {
                    const uint4* vt = reinterpret_cast<const uint4*>(sm.tchunk(st, lc));
                    float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
                    for (int v = 0; v < NV; ++v) {
                        float xs[E];
                        EL::unpack(vt[v * 32 + lane], xs);
#pragma unroll
                        for (int e = 0; e < E; ++e)
                            acc[e & 3] += weight(xs[e], m_t, c);
                    }
                    const double pc = warp_sum((double)((acc[0] + acc[1]) + (acc[2] + acc[3])));
                    if (lane == 0)
                        a.Pc[trow * a.nchunks + (c0 + lc)] = pc;
                    wst += pc;
                    if (dc.use_draft) {
                        const uint4* vd = reinterpret_cast<const uint4*>(sm.dchunk(st, lc));
                        float accd[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
                        for (int v = 0; v < NV; ++v) {
                            float xs[E];
                            EL::unpack(vd[v * 32 + lane], xs);
#pragma unroll
                            for (int e = 0; e < E; ++e)
                                accd[e & 3] += weight(xs[e], m_d, c);
                        }
                        wsd += warp_sum((double)((accd[0] + accd[1]) + (accd[2] + accd[3])));
                    }
                }
            }
            if (lane == 0) {
                s_wsum[warp][0] = wst;
                s_wsum[warp][1] = wsd;
            }
            __syncthreads();
            if (tid < C) {
                double s0 = 0.0, s1 = 0.0;
                for (int w = 0; w < nw; ++w) {
                    s0 += s_wsum[w][0];
                    s1 += s_wsum[w][1];
                }
                const uint32_t dst = map_to_rank(smem_addr(&s_csum[rank][0]), (uint32_t)tid);
                st_cluster_f64(dst, s0);
                st_cluster_f64(dst + 8, s1);
            }
            cluster_arrive();
            cluster_wait();   // C
            double St = 0.0, Sd = 0.0;
            for (int r = 0; r < C; ++r) {
                St += s_csum[r][0];
                Sd += s_csum[r][1];
            }
            const bool row_ok = work && St > 0.0 && (!dc.use_draft || Sd > 0.0);
            const float inv_st = row_ok ? (float)(1.0 / St) : 0.0f;
            const float inv_sd = row_ok && dc.use_draft ? (float)(1.0 / Sd) : 0.0f;
            bool accept = false;
            float px = NAN, qx = NAN;
            if (dc.is_test && row_ok) {
                const T* tg = static_cast<const T*>(a.tgt) + trow * (size_t)V;
                const T* dg = static_cast<const T*>(a.drf) + ((size_t)dc.b * Kmax + dc.i) * (size_t)V;
                const float et = weight(EL::load(tg + dc.x), m_t, c);
                const float ed = weight(EL::load(dg + dc.x), m_d, c);
                px = __fmul_rn(et, inv_st);
                qx = __fmul_rn(ed, inv_sd);
                accept = __fmul_rn(dc.u, qx) < px;   // u < min(1, p/q) without a division
            }
            const uint8_t d = !row_ok ? kDecInvalid
                                      : (dc.is_test ? (accept ? kDecAccept : kDecReject) : kDecBonus);
            if (rank == 0 && tid == 0) {
                if (dc.is_test && d != kDecAccept)
                    atomicOr(a.mask + dc.b, 1u << dc.i);
                a.dec[trow] = d;
                a.rowstat[trow] = make_float4(m_t, inv_st, m_d, inv_sd);
                if (dc.is_test && a.p_x) {
                    a.p_x[(size_t)dc.b * Kmax + dc.i] = px;
                    a.q_x[(size_t)dc.b * Kmax + dc.i] = qx;
                }
            }
            // ---- pass 3: residual mass per chunk of rows that may be drawn from ----
            if (dc.use_draft && row_ok && (d == kDecReject || !a.early_exit)) {
                for (int lc = warp; lc < nck; lc += nw) {
                    const uint4* vt = reinterpret_cast<const uint4*>(sm.tchunk(st, lc));
                    const uint4* vd = reinterpret_cast<const uint4*>(sm.dchunk(st, lc));
                    float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
                    for (int v = 0; v < NV; ++v) {
                        float xt[E], xd[E];
                        EL::unpack(vt[v * 32 + lane], xt);
                        EL::unpack(vd[v * 32 + lane], xd);
#pragma unroll
                        for (int e = 0; e < E; ++e)
                            acc[e & 3] += resid_term(weight(xt[e], m_t, c), inv_st,
                                                     weight(xd[e], m_d, c), inv_sd);
                    }
                    const double rc = warp_sum((double)((acc[0] + acc[1]) + (acc[2] + acc[3])));
                    if (lane == 0)
                        a.Rc[trow * a.nchunks + (c0 + lc)] = rc;
                }
            }
        }
        if (s_bad && !poisoned_before && tid == 0)
            atomicOr(a.err, kErrWaitTimeout);
        __syncthreads();   // stage st fully consumed
        if (stages == 1 && dn.idx >= 0)
            issue_row<T, NV>(a, sm, dn, 0, c0, nck, warp, nw, lane, s_bad != 0);
        dc = dn;
        dn = dnn;
    }
}

}  // namespace sv
