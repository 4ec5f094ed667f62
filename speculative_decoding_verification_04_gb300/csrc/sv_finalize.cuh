// sv_finalize.cuh -- per-sequence finalisation, one warp per sequence.
//
// Runs after the sweep (programmatic dependent launch: it waits on
// griddepcontrol.wait before touching the sweep's results).  For sequence b:
//   * warp ballot over the per-position decisions: n = index of the first
//     position that was not accepted (K_b if all were) -- the first-rejection
//     reduction;
//   * greedy: the token is the argmax of row n;
//   * sampling: the distribution of row n is the residual max(0, p - q)
//     (n < K_b) or p itself (n = K_b).  A fp64 prefix over its per-chunk sums
//     picks the chunk holding u * S; that one chunk of logits is re-read, its
//     terms recomputed with the sweep's exact rounding sequence, and an
//     in-chunk prefix scan finds the smallest j with u * S < C_j;
//   * outputs: accepted draft tokens, the drawn token, -1 padding, n.
#pragma once

#include "sv_common.cuh"

namespace sv {

// Inverse-CDF draw from row n of sequence b (whole warp; every lane returns
// the same token, or -1 if nothing can be drawn).
template <typename T, int NV>
__device__ int draw_token(const Args& a, int b, int Kb, float Tb, int n, float uf, int lane)
{
    using EL = Elem<T>;
    constexpr int CH = 32 * NV * EL::E;
    constexpr int L = CH / 32;   // contiguous elements per lane in the chunk scan
    const int nchunks = a.nchunks;
    const size_t r = (size_t)b * (a.Kmax + 1) + n;
    bool resid = n < Kb && a.has_draft != 0;
    const int per = (nchunks + 31) / 32;
    const int lo = min(nchunks, lane * per), hi = min(nchunks, lo + per);
    int chunk = -1;
    double tloc = 0.0;
    for (int attempt = 0; attempt < 2 && chunk < 0; ++attempt) {
        const float* sums = (resid ? a.Rc : a.Pc) + r * nchunks;
        double ls = 0.0;
        for (int c = lo; c < hi; ++c)
            ls += (double)__ldcg(sums + c);
        const double inc = warp_incl_scan(ls, lane);
        const double S = __shfl_sync(kFull, inc, 31);
        const double up = __shfl_up_sync(kFull, inc, 1);
        const double excl = lane == 0 ? 0.0 : up;
        if (!(S > 0.0) || !isfinite(S)) {
            if (resid) {   // zero residual mass: draw from p of the same row
                resid = false;
                continue;
            }
            break;
        }
        const double t = (double)uf * S;
        int cand = -1, lastpos = -1;
        double cum = excl, bcand = 0.0, blast = 0.0;
        for (int c = lo; c < hi; ++c) {
            const double s = (double)__ldcg(sums + c);
            const double before = cum;
            cum += s;
            if (s > 0.0) {
                lastpos = c;
                blast = before;
            }
            if (cand < 0 && t < cum) {
                cand = c;
                bcand = before;
            }
        }
        double before_sel = 0.0;
        const unsigned has = __ballot_sync(kFull, cand >= 0);
        if (has) {
            const int src = __ffs(has) - 1;
            chunk = __shfl_sync(kFull, cand, src);
            before_sel = __shfl_sync(kFull, bcand, src);
        } else {
            const unsigned pos = __ballot_sync(kFull, lastpos >= 0);
            if (pos) {
                const int src = 31 - __clz(pos);
                chunk = __shfl_sync(kFull, lastpos, src);
                before_sel = __shfl_sync(kFull, blast, src);
            }
        }
        tloc = t - before_sel;
    }
    if (chunk < 0)
        return -1;

    const float4 st = __ldcg(a.rowstat + r);   // m_t, 1/S_t, m_d, 1/S_d
    const float c = log2e_over(Tb);
    const T* tg = static_cast<const T*>(a.tgt) + r * (size_t)a.V;
    const T* dg = resid ? static_cast<const T*>(a.drf) + ((size_t)b * a.Kmax + n) * (size_t)a.V
                        : nullptr;
    const int e0 = chunk * CH;
    const int len = min(CH, a.V - e0);
    const int j0 = min(len, lane * L), j1 = min(len, j0 + L);
    auto value = [&](int j) -> float {
        const float et = weight(EL::load(tg + e0 + j), st.x, c);
        if (!resid)
            return et;
        return resid_term(et, st.y, weight(EL::load(dg + e0 + j), st.z, c), st.w);
    };
    // lane-contiguous spans: compensated fp32 sums, fp64 scan across lanes
    CompSum span;
    int lastpos = -1;
    for (int j = j0; j < j1; ++j) {
        const float v = value(j);
        span.add(v);
        if (v > 0.0f)
            lastpos = j;
    }
    const double ls = (double)span.s + (double)span.c;
    const double inc = warp_incl_scan(ls, lane);
    const double up = __shfl_up_sync(kFull, inc, 1);
    const double excl = lane == 0 ? 0.0 : up;
    // the mass this lane's span must still cover, small enough for fp32
    const float t_lane = (float)(tloc - excl);
    int cand = INT_MAX;
    if (t_lane < (float)ls) {   // spans before the target lane cannot hold it
        CompSum cum;
        for (int j = j0; j < j1; ++j) {
            cum.add(value(j));
            if (t_lane < cum.value()) {
                cand = j;
                break;
            }
        }
    }
    const int best = __reduce_min_sync(kFull, cand);
    const int last = __reduce_max_sync(kFull, lastpos);
    if (best != INT_MAX)
        return e0 + best;
    return last >= 0 ? e0 + last : -1;
}

template <typename T, int NV>
__global__ void __launch_bounds__(kFinalizeWarps * 32) sv_finalize_kernel(const Args a)
{
    griddep_wait();   // the sweep has completed and its writes are visible
    const int lane = threadIdx.x & 31;
    const int b = blockIdx.x * kFinalizeWarps + (int)(threadIdx.x >> 5);
    if (b >= a.B)
        return;
    const int Kb = __ldg(a.K + b);
    const float Tb = __ldg(a.temp + b);
    const bool greedy = Tb == 0.0f;
    const size_t rb = (size_t)b * (a.Kmax + 1);

    // first-rejection reduction: one warp ballot over the K_b <= 32 decisions
    const uint8_t d = lane < Kb ? ld_cg_u8(a.dec + rb + lane) : (uint8_t)kDecAccept;
    const unsigned notacc = __ballot_sync(kFull, d != kDecAccept);
    const int n = notacc ? __ffs(notacc) - 1 : Kb;
    bool bad = !temperature_usable(Tb);
    const uint8_t dn = ld_cg_u8(a.dec + rb + n);
    bad = bad || (n < Kb ? dn != kDecReject : dn != kDecBonus);
    float uf = 0.0f;
    if (!greedy) {
        uf = __ldg(a.uni + (size_t)b * (a.Kmax + 1) + Kb);
        bad = bad || !(uf >= 0.0f && uf < 1.0f);
    }
    int token = -1;
    if (!bad)
        token = greedy ? __ldcg(a.argmax + rb + n) : draw_token<T, NV>(a, b, Kb, Tb, n, uf, lane);
    bad = bad || token < 0 || token >= a.V;

    int32_t* orow = a.out_tok + rb;
    for (int j = lane; j <= a.Kmax; j += 32)
        orow[j] = bad ? -1 : (j < n ? __ldg(a.tok + (size_t)b * a.Kmax + j) : (j == n ? token : -1));
    if (lane == 0) {
        a.out_n[b] = bad ? -1 : n;
        if (a.want_final)
            a.final_row[b] = bad ? -1 : n;
    }
    if (a.want_resid) {
        for (int i = lane; i < a.Kmax; i += 32) {
            float v = NAN;
            if (!greedy && i < Kb) {
                const uint8_t di = ld_cg_u8(a.dec + rb + i);
                if (di == kDecAccept || di == kDecReject) {
                    const float* rc = a.Rc + (rb + i) * a.nchunks;
                    double s = 0.0;
                    for (int c = 0; c < a.nchunks; ++c)
                        s += (double)__ldcg(rc + c);
                    v = (float)s;
                }
            }
            a.resid[(size_t)b * a.Kmax + i] = v;
        }
    }
}

}  // namespace sv
