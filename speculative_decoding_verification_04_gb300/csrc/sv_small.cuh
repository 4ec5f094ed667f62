// sv_small.cuh -- verification for small vocabularies (V <= kSmallVocab): one
// warp per sequence, each row held in the warp's registers (lane l: elements
// l, l + 32, l + 64, ...), no shared memory, no clusters.  For such rows the
// cluster sweep's per-row exchange and copy latency dwarf the work; here many
// sequences are in flight at once, one per warp.
//
// The operation is the sweep's (and the pages'): at a tested sampling row p
// and q are weighed against the row maxima (rows this small need no
// reference trick), accept iff u q(x) < p(x); at the sequence's final row the
// token is drawn by inverse CDF from normalize(max(0, p - q)) (a rejection;
// p when it has no mass) or from p (the bonus row); greedy rows keep x iff it
// is the lowest index holding the row maximum.  Unusable input on the walk
// gives -1 outputs.  Sums are fp32 with compensation (TwoSum) within and
// across lanes.
#pragma once

#include "sv_sweep.cuh"

namespace sv {

constexpr int kSmallVocab = 1024;   // largest V the warp kernel takes

// Row `row` of V elements into the lane's NE registers (-inf past V).
template <typename T, int NE>
__device__ __forceinline__ void small_load(const T* row, int V, int lane, float (&x)[NE])
{
#pragma unroll
    for (int e = 0; e < NE; ++e) {
        const int j = e * 32 + lane;
        x[e] = j < V ? Elem<T>::load(row + j) : -INFINITY;
    }
}

// The row's maximum (every lane); `bad` when it holds a NaN or +inf or has
// no finite entry (a row the method cannot use).
template <int NE>
__device__ __forceinline__ float small_max(const float (&x)[NE], bool& bad)
{
    float m = -INFINITY;
    bool b = false;
#pragma unroll
    for (int e = 0; e < NE; ++e) {
        b = b || isnan(x[e]) || x[e] == INFINITY;
        m = fmaxf(m, x[e]);
    }
    b = __any_sync(kFull, b);
    m = warp_max_nan(m);
    bad = b || !(m > -INFINITY);
    return m;
}

// w[e] = exp2(fma(x[e], c, -r)) (the sweep's weight), and their warp sum,
// compensated within the lane and across the warp.
template <int NE>
__device__ __forceinline__ float small_weights(const float (&x)[NE], float r, float c, float (&w)[NE])
{
    float s = 0.0f, cmp = 0.0f;
#pragma unroll
    for (int e = 0; e < NE; ++e) {
        w[e] = weight_r(x[e], r, c);
        float t, er;
        two_sum(s, w[e], t, er);
        s = t;
        cmp += er;
    }
    return warp_sum_comp(s + cmp);
}

// Element x (0 <= x < 32 NE) of a lane-interleaved row, in every lane.
template <int NE>
__device__ __forceinline__ float small_at(const float (&v)[NE], int x)
{
    float r = 0.0f;
#pragma unroll
    for (int e = 0; e < NE; ++e)
        r = (e == (x >> 5)) ? v[e] : r;
    return __shfl_sync(kFull, r, x & 31);
}

// The lowest index holding the row maximum (every lane).
template <int NE>
__device__ __forceinline__ int small_argmax(const float (&x)[NE], int lane)
{
    float lm = -INFINITY;
    int li = INT_MAX;
#pragma unroll
    for (int e = 0; e < NE; ++e)
        if (x[e] > lm) {   // strictly greater: the lane's lowest index keeps a tie
            lm = x[e];
            li = e * 32 + lane;
        }
    const float m = warp_max_nan(lm);
    return __reduce_min_sync(kFull, lm == m ? li : INT_MAX);
}

// Inverse CDF over non-negative masses a (lane-interleaved, index order e
// then lane): the smallest j with u S < a_0 + ... + a_j, prefix sums
// compensated; beyond the total (rounding) the last element with mass; -1 if
// none has mass.  Every lane gets the result, and `near`: the point u S lies
// within 1e-6 S of a bound of the element taken (always so beyond the total).
template <int NE>
__device__ __forceinline__ int small_draw(const float (&a)[NE], float S, float u, int lane, bool& near)
{
    const float t = u * S;
    float base_s = 0.0f, base_c = 0.0f;
    int last_pos = -1;
#pragma unroll
    for (int e = 0; e < NE; ++e) {
        const float d = a[e];
        if (d > 0.0f)
            last_pos = e * 32 + lane;
        float s, cc;
        warp_incl_scan_comp(d, lane, s, cc);
        const float rel = (t - base_s) - base_c;
        const unsigned hit = __ballot_sync(kFull, d > 0.0f && rel < s + cc);
        if (hit) {
            const int src = __ffs(hit) - 1;
            const float dist = fminf(rel - ((s + cc) - d), (s + cc) - rel);   // in lane src
            near = __shfl_sync(kFull, dist < 1e-6f * S ? 1 : 0, src) != 0;
            return e * 32 + src;
        }
        const float gs = __shfl_sync(kFull, s, 31), gc = __shfl_sync(kFull, cc, 31);
        float ts, te;
        two_sum(base_s, gs, ts, te);
        base_s = ts;
        base_c += gc + te;
    }
    near = true;
    return __reduce_max_sync(kFull, last_pos);
}

// One warp per sequence.  A warp takes `tile` consecutive sequences at a time
// (so that K, the row starts and the temperatures load in one coalesced
// read), then the tile a grid's worth of warps further on; tile = 1 when the
// batch is no larger than the grid's warps.
template <typename T, int NE>
__global__ void __launch_bounds__(128, 4) sv_small_kernel(const Args a)
{
    const int lane = threadIdx.x & 31;
    const int warp = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
    const int nwarps = (int)((gridDim.x * blockDim.x) >> 5);
    const int V = a.V, Kmax = a.Kmax, tile = a.small_tile;
    const T* tgt = static_cast<const T*>(a.tgt);
    const T* drf = static_cast<const T*>(a.drf);
    uint32_t c_seq = 0, c_inv = 0, c_test = 0, c_acc = 0, c_commit = 0, c_tie = 0, c_dtie = 0;   // lane 0
    const bool want_diag = a.want_pq || a.want_resid;

    for (long long b0 = (long long)warp * tile; b0 < a.B; b0 += (long long)nwarps * tile) {
        const int ns = (int)min((long long)tile, (long long)a.B - b0);
        const int bl = (int)b0 + lane;
        const bool in = lane < ns;
        const int Kl = in ? __ldg(a.K + bl) : 0;
        const float Tl = in ? __ldg(a.temp + bl) : 0.0f;
        const int tbl = in ? (a.packed ? __ldg(a.cu_t + bl) : bl * (Kmax + 1)) : 0;
        const int dbl = in ? (a.packed ? __ldg(a.cu_d + bl) : bl * Kmax) : 0;
        for (int s = 0; s < ns; ++s) {
            const int b = (int)b0 + s;
            const int Kb = __shfl_sync(kFull, Kl, s);
            const float Tb = __shfl_sync(kFull, Tl, s);
            const int tb = __shfl_sync(kFull, tbl, s);
            const int db = __shfl_sync(kFull, dbl, s);
            // the sequence's draft tokens and test uniforms, lane j: position
            // j (K_b <= 32); the final draw's uniform (slot K_b, which may be 32)
            const int tokj = lane < Kmax ? __ldg(a.tok + (size_t)b * Kmax + lane) : 0;
            const float unij = lane < Kmax ? __ldg(a.uni + (size_t)b * (Kmax + 1) + lane) : 0.0f;
            const float uf = (Tb != 0.0f && Kb >= 0 && Kb <= Kmax) ? __ldg(a.uni + (size_t)b * (Kmax + 1) + Kb) : 0.0f;
            const bool greedy = Tb == 0.0f;
            bool bad = !temperature_usable(Tb);
            const float c = (!bad && !greedy) ? log2e_over(Tb) : 0.0f;
            int n = -1, token = -1;   // the outputs, once the walk stops
            bool dnear = false;       // the final draw's point near a bound of its token
            int next_pos = 0;         // diagnostics written for positions below it
            // the walk; after its stop, rows are read only for diagnostics
            // (verify-all), as long as they are usable
            for (int i = 0; !bad && i <= Kb; ++i) {
                const bool test = i < Kb;
                const bool stopped = n >= 0;
                if (stopped && (greedy || !test || a.early_exit))
                    break;
                const size_t pos = (size_t)b * Kmax + i;
                float at[NE];   // the target row; its weights once weighed
                small_load<T, NE>(tgt + ((size_t)tb + i) * (size_t)V, V, lane, at);
                bool rbad = false;
                const float mt = small_max<NE>(at, rbad);
                if (greedy) {
                    const int g = small_argmax<NE>(at, lane);
                    const int x = __shfl_sync(kFull, tokj, i & 31);
                    if (rbad || g >= V || (test && (x < 0 || x >= V))) {
                        bad = true;
                        break;
                    }
                    if (test && lane == 0 && a.want_stats) {
                        ++c_test;
                        c_acc += x == g ? 1u : 0u;
                    }
                    if (test && x == g)
                        continue;
                    n = i;
                    token = g;
                    break;
                }
                // sampling
                const int x = __shfl_sync(kFull, tokj, i & 31);
                const float u = __shfl_sync(kFull, unij, i & 31);
                if (rbad || (test && (!a.has_draft || x < 0 || x >= V || !(u >= 0.0f && u < 1.0f)))) {
                    bad = !stopped;
                    break;
                }
                const float St = small_weights<NE>(at, ref_of(mt, c), c, at);
                if (!(St > 0.0f && isfinite(St))) {
                    bad = !stopped;
                    break;
                }
                const float ist = __frcp_rn(St);
                if (!test) {   // the bonus row: the token from p
                    if (!(uf >= 0.0f && uf < 1.0f)) {
                        bad = true;
                        break;
                    }
                    n = i;
                    token = small_draw<NE>(at, St, uf, lane, dnear);
                    break;
                }
                float ad[NE];   // the draft row; its weights; then the residual
                small_load<T, NE>(drf + ((size_t)db + i) * (size_t)V, V, lane, ad);
                bool dbad = false;
                const float md = small_max<NE>(ad, dbad);
                const float Sd = dbad ? 0.0f : small_weights<NE>(ad, ref_of(md, c), c, ad);
                if (dbad || !(Sd > 0.0f && isfinite(Sd))) {
                    bad = !stopped;
                    break;
                }
                const float isd = __frcp_rn(Sd);
                const float px = __fmul_rn(small_at<NE>(at, x), ist);
                const float qx = __fmul_rn(small_at<NE>(ad, x), isd);
                const bool accept = __fmul_rn(u, qx) < px;   // u < min(1, p/q) without a division
                if (lane == 0 && a.want_pq) {
                    a.p_x[pos] = px;
                    a.q_x[pos] = qx;
                }
                if (!stopped && lane == 0 && a.want_stats) {
                    ++c_test;
                    c_acc += accept ? 1u : 0u;
                    c_tie += fabsf(__fmaf_rn(u, qx, -px)) < 1e-6f * qx ? 1u : 0u;
                }
                next_pos = i + 1;
                if (accept && !want_diag && a.early_exit)
                    continue;
                // the residual max(0, p - q), over the draft's weights
                float rs = 0.0f, rc = 0.0f;
#pragma unroll
                for (int e = 0; e < NE; ++e) {
                    ad[e] = fmaxf(__fsub_rn(__fmul_rn(at[e], ist), __fmul_rn(ad[e], isd)), 0.0f);
                    float t, er;
                    two_sum(rs, ad[e], t, er);
                    rs = t;
                    rc += er;
                }
                const float SR = warp_sum_comp(rs + rc);
                if (lane == 0 && a.want_resid)
                    a.resid[pos] = SR;
                if (!stopped && !accept) {
                    if (!(uf >= 0.0f && uf < 1.0f)) {
                        bad = true;
                        break;
                    }
                    n = i;
                    // no residual mass (p and q equal to rounding): p of the row
                    token = SR > 0.0f ? small_draw<NE>(ad, SR, uf, lane, dnear)
                                      : small_draw<NE>(at, St, uf, lane, dnear);
                }
            }
            if (bad)
                n = -1;
            // positions without diagnostics (greedy, unreached, past K_b) carry NaN
            if (want_diag && lane == 0)
                for (int i = greedy ? 0 : next_pos; i < Kmax; ++i) {
                    const size_t pos = (size_t)b * Kmax + i;
                    if (a.want_pq) {
                        a.p_x[pos] = NAN;
                        a.q_x[pos] = NAN;
                    }
                    if (a.want_resid)
                        a.resid[pos] = NAN;
                }
            // outputs (and the KV length), counters
            const bool ok = !bad && n >= 0 && token >= 0 && token < V;
            int32_t* orow = a.out_tok + (size_t)b * (Kmax + 1);
            for (int j = lane; j <= Kmax; j += 32)
                orow[j] = !ok ? -1 : (j < n ? tokj : (j == n ? token : -1));
            if (lane == 0) {
                a.out_n[b] = ok ? n : -1;
                if (a.want_final)
                    a.final_row[b] = ok ? n : -1;
                if (a.want_kv && ok)
                    a.kv_len[b] += n + 1;
                if (ok) {
                    ++c_seq;
                    c_commit += (uint32_t)n + 1u;
                    c_dtie += dnear ? 1u : 0u;
                } else {
                    ++c_inv;
                }
            }
        }
    }
    if (a.want_stats && lane == 0) {
        const uint32_t cs[7] = {c_seq, c_inv, c_test, c_acc, c_commit, c_tie, c_dtie};
#pragma unroll
        for (int k = 0; k < 7; ++k)
            if (cs[k])
                atomicAdd(a.stats + k, (unsigned long long)cs[k]);
    }
}

}  // namespace sv
