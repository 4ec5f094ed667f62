// spec_verify.cu -- libspecverify: batched draft-token verification by
// modified rejection sampling on one GB300 (sm_103a).
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
// GB300 design (one fused launch per call):
//  * One thread-block cluster of C CTAs per (position i, sequence b) row,
//    clusters ordered position-major so that position 0 of every sequence is
//    swept first.  Each CTA owns `ncpc` contiguous vocabulary chunks of the
//    target row (and of the draft row for tested sampling positions) and
//    stages them into shared memory with 1-D bulk copies (cp.async.bulk, one
//    mbarrier per chunk).  The row stays resident for every later pass.
//  * Pass 1 (as chunks land): NaN-propagating max, warp shuffles, cluster
//    all-reduce through distributed shared memory.
//  * Pass 2: sum of exp2((l - m) * log2(e)/T) per chunk (fp32 per lane, fp64
//    across lanes), chunk sums written out, cluster all-reduce of S.  Greedy
//    rows instead find the lowest index holding the max.
//  * Decision: p(x) * (u q(x) < p(x)), by every CTA identically; a rejection
//    sets a per-sequence bit so later positions of that sequence skip their
//    rows entirely (the method never reads them).
//  * Pass 3 (rejected rows only): per-chunk residual mass
//    sum max(0, p - q), from the resident row.
//  * The last CTA of a sequence to arrive (atomic counter, no spin-wait)
//    finalises it: warp ballot over the accept decisions gives nacc, a
//    prefix over the chunk sums of row nacc picks the chunk, one chunk of
//    logits is re-read and scanned to draw the token by inverse CDF.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <limits.h>

#include <map>
#include <mutex>
#include <tuple>
#include <vector>

#include "../../include/specverify.h"
#include "sv_ptx.cuh"

namespace sv {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kMaxWarps = 16;
constexpr int kMaxCluster = 16;
constexpr uint32_t kWaitSpins = 1u << 22;   // bounded mbarrier polls (seconds)
constexpr double kLog2e = 1.4426950408889634;

enum : uint8_t {
    kDecNone = 0,      // row not evaluated in this call
    kDecAccept = 1,
    kDecReject = 2,
    kDecInvalid = 3,   // unusable input on this row
    kDecBonus = 4      // position K_b evaluated and usable
};

enum : uint32_t { kErrWaitTimeout = 1u };

struct Args {
    const void* tgt;
    const void* drf;
    const int32_t* tok;
    const float* uni;
    const float* temp;
    int32_t* out_tok;
    int32_t* out_n;
    int B, Kmax, V;
    int nchunks, ncpc, C;
    int early_exit, aligned;
    // workspace
    uint32_t* err;
    int* counter;
    uint32_t* mask;
    uint8_t* dec;
    const int32_t* K;
    int32_t* argmax;
    float4* rowstat;
    double* Pc;   // per (row, chunk): sum of exp2((l - m_t) c) over the chunk
    double* Rc;   // per (row, chunk): sum of max(0, p - q) over the chunk
    // diagnostics (nullable)
    float* p_x;
    float* q_x;
    float* resid;
    int32_t* final_row;
};

// ---------------------------------------------------------------------------
// element access
// ---------------------------------------------------------------------------
template <typename T> struct Elem;

template <> struct Elem<float> {
    static constexpr int E = 4;   // elements per 16-byte vector
    __device__ static __forceinline__ void unpack(const uint4& w, float (&x)[4])
    {
        x[0] = __uint_as_float(w.x);
        x[1] = __uint_as_float(w.y);
        x[2] = __uint_as_float(w.z);
        x[3] = __uint_as_float(w.w);
    }
    __device__ static __forceinline__ float load(const float* p) { return __ldg(p); }
    __device__ static __forceinline__ void copy(float* dst, const float* src) { *dst = __ldg(src); }
    __device__ static __forceinline__ void set_neg_inf(float* dst) { *dst = -INFINITY; }
};

template <> struct Elem<__nv_bfloat16> {
    static constexpr int E = 8;
    __device__ static __forceinline__ void unpack(const uint4& w, float (&x)[8])
    {
        const uint32_t v[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            x[2 * k] = __uint_as_float(v[k] << 16);
            x[2 * k + 1] = __uint_as_float(v[k] & 0xffff0000u);
        }
    }
    __device__ static __forceinline__ float load(const __nv_bfloat16* p)
    {
        const unsigned short h = __ldg(reinterpret_cast<const unsigned short*>(p));
        return __uint_as_float(static_cast<uint32_t>(h) << 16);
    }
    __device__ static __forceinline__ void copy(__nv_bfloat16* dst, const __nv_bfloat16* src)
    {
        *reinterpret_cast<unsigned short*>(dst) = __ldg(reinterpret_cast<const unsigned short*>(src));
    }
    __device__ static __forceinline__ void set_neg_inf(__nv_bfloat16* dst)
    {
        *reinterpret_cast<unsigned short*>(dst) = 0xFF80u;
    }
};

// exp2((l - m) * c), the unnormalised softmax weight, in one fixed rounding
// sequence shared by every pass and by the finaliser.
__device__ __forceinline__ float weight(float l, float m, float c)
{
    return ex2_approx(__fmul_rn(__fsub_rn(l, m), c));
}

// max(0, p - q) with p = e_t / S_t, q = e_d / S_d (one fixed rounding sequence).
__device__ __forceinline__ float resid_term(float et, float inv_st, float ed, float inv_sd)
{
    return fmaxf(__fsub_rn(__fmul_rn(et, inv_st), __fmul_rn(ed, inv_sd)), 0.0f);
}

__device__ __forceinline__ float warp_max_nan(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v = max_nan(v, __shfl_xor_sync(kFull, v, o));
    return v;
}

// Butterfly sum: every lane ends with the same value (IEEE addition commutes).
__device__ __forceinline__ double warp_sum(double v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v += __shfl_xor_sync(kFull, v, o);
    return v;
}

__device__ __forceinline__ double warp_incl_scan(double v, int lane)
{
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const double y = __shfl_up_sync(kFull, v, o);
        if (lane >= o)
            v += y;
    }
    return v;
}

__device__ __forceinline__ bool temperature_usable(float T)
{
    return T == 0.0f || (isfinite(T) && T >= FLT_MIN);
}

// ---------------------------------------------------------------------------
// final draw for one sequence (whole CTA)
// ---------------------------------------------------------------------------
// Returns the drawn token of row n of sequence b, or -1 if it cannot be drawn.
template <typename T, int NV>
__device__ __noinline__ int draw_final_token(const Args& a, int b, int Kb, float Tb, int n)
{
    using EL = Elem<T>;
    constexpr int CH = 32 * NV * EL::E;
    __shared__ int f_chunk, f_resid;
    __shared__ double f_tloc;
    __shared__ double f_wtot[kMaxWarps];
    __shared__ int f_wcand[kMaxWarps], f_wlast[kMaxWarps];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
    const int nchunks = a.nchunks;
    const size_t r = (size_t)b * (a.Kmax + 1) + n;

    // Chunk selection by one warp: lane-contiguous chunk ranges, fp64 prefix.
    if (warp == 0) {
        bool resid = n < Kb;
        const int per = (nchunks + 31) / 32;
        const int lo = min(nchunks, lane * per), hi = min(nchunks, lo + per);
        const double uf = (double)a.uni[(size_t)b * (a.Kmax + 1) + Kb];
        int chunk = -1;
        double before_sel = 0.0;
        for (int attempt = 0; attempt < 2 && chunk < 0; ++attempt) {
            const double* sums = (resid ? a.Rc : a.Pc) + r * nchunks;
            double ls = 0.0;
            for (int c = lo; c < hi; ++c)
                ls += __ldcg(sums + c);
            const double inc = warp_incl_scan(ls, lane);
            const double S = __shfl_sync(kFull, inc, 31);
            const double up = __shfl_up_sync(kFull, inc, 1);
            const double excl = lane == 0 ? 0.0 : up;
            if (!(S > 0.0) || !isfinite(S)) {
                if (resid) {          // zero residual mass: draw from p of this row
                    resid = false;
                    continue;
                }
                break;                // nothing to draw from
            }
            const double t = uf * S;
            int cand = -1, lastpos = -1;
            double cum = excl, bcand = 0.0, blast = 0.0;
            for (int c = lo; c < hi; ++c) {
                const double s = __ldcg(sums + c);
                const double before = cum;
                cum += s;
                if (s > 0.0) { lastpos = c; blast = before; }
                if (cand < 0 && t < cum) { cand = c; bcand = before; }
            }
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
            if (chunk >= 0 && lane == 0) {
                f_tloc = t - before_sel;
                f_resid = resid ? 1 : 0;
            }
        }
        if (lane == 0)
            f_chunk = chunk;
    }
    __syncthreads();
    const int chunk = f_chunk;
    if (chunk < 0)
        return -1;
    const bool resid = f_resid != 0;
    const double tloc = f_tloc;

    const float4 st = __ldcg(a.rowstat + r);   // m_t, 1/S_t, m_d, 1/S_d
    const float c = (float)(kLog2e / (double)Tb);
    const T* tg = static_cast<const T*>(a.tgt) + r * (size_t)a.V;
    const T* dg = resid ? static_cast<const T*>(a.drf) + ((size_t)b * a.Kmax + n) * (size_t)a.V
                        : nullptr;
    const long long e0 = (long long)chunk * CH;
    const int len = (int)min((long long)CH, (long long)a.V - e0);
    const int per_t = (len + blockDim.x - 1) / blockDim.x;
    const int j0 = min(len, tid * per_t), j1 = min(len, j0 + per_t);

    auto value = [&](int j) -> float {
        const float et = weight(EL::load(tg + e0 + j), st.x, c);
        if (!resid)
            return et;
        const float ed = weight(EL::load(dg + e0 + j), st.z, c);
        return resid_term(et, st.y, ed, st.w);
    };

    double ls = 0.0;
    int lastpos = -1;
    for (int j = j0; j < j1; ++j) {
        const float v = value(j);
        ls += (double)v;
        if (v > 0.0f)
            lastpos = j;
    }
    // block exclusive scan of the per-thread sums
    const double inc = warp_incl_scan(ls, lane);
    const double up = __shfl_up_sync(kFull, inc, 1);
    if (lane == 31)
        f_wtot[warp] = inc;
    __syncthreads();
    double excl = lane == 0 ? 0.0 : up;
    for (int w = 0; w < warp; ++w)
        excl += f_wtot[w];
    int cand = INT_MAX;
    double cum = excl;
    for (int j = j0; j < j1; ++j) {
        cum += (double)value(j);
        if (tloc < cum) {
            cand = j;
            break;
        }
    }
    const int wc = __reduce_min_sync(kFull, cand);
    const int wl = __reduce_max_sync(kFull, lastpos);
    if (lane == 0) {
        f_wcand[warp] = wc;
        f_wlast[warp] = wl;
    }
    __syncthreads();
    int best = INT_MAX, last = -1;
    for (int w = 0; w < nw; ++w) {
        best = min(best, f_wcand[w]);
        last = max(last, f_wlast[w]);
    }
    __syncthreads();   // f_* are reused by the next sequence this CTA finalises
    if (best != INT_MAX)
        return (int)(e0 + best);
    return last >= 0 ? (int)(e0 + last) : -1;
}

// ---------------------------------------------------------------------------
// per-sequence finalisation (whole CTA, last arrival of the sequence)
// ---------------------------------------------------------------------------
template <typename T, int NV>
__device__ __noinline__ void finalize_sequence(const Args& a, int b, int Kb, float Tb)
{
    __shared__ int f_n, f_bad;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const size_t rb = (size_t)b * (a.Kmax + 1);
    const bool greedy = (Tb == 0.0f);

    if (warp == 0) {
        // warp ballot over the accept decisions: nacc = first non-accept
        const uint8_t d = lane < Kb ? ld_cg_u8(a.dec + rb + lane) : (uint8_t)kDecAccept;
        const unsigned notacc = __ballot_sync(kFull, d != kDecAccept);
        const int n = notacc ? __ffs(notacc) - 1 : Kb;
        if (lane == 0) {
            int bad = !temperature_usable(Tb);
            const uint8_t dn = ld_cg_u8(a.dec + rb + n);
            bad |= (n < Kb) ? (dn != kDecReject) : (dn != kDecBonus);
            if (!greedy) {
                const float uf = a.uni[(size_t)b * (a.Kmax + 1) + Kb];
                bad |= !(uf >= 0.0f && uf < 1.0f);
            }
            f_n = n;
            f_bad = bad;
        }
    }
    __syncthreads();
    const int n = f_n;
    int token = -1;
    if (!f_bad) {
        if (greedy)
            token = __ldcg(a.argmax + rb + n);
        else
            token = draw_final_token<T, NV>(a, b, Kb, Tb, n);
    }
    const bool bad = f_bad || token < 0 || token >= a.V;
    int32_t* orow = a.out_tok + (size_t)b * (a.Kmax + 1);
    for (int j = tid; j <= a.Kmax; j += blockDim.x)
        orow[j] = bad ? -1 : (j < n ? a.tok[(size_t)b * a.Kmax + j] : (j == n ? token : -1));
    if (tid == 0) {
        a.out_n[b] = bad ? -1 : n;
        if (a.final_row)
            a.final_row[b] = bad ? -1 : n;
    }
    if (a.resid) {
        for (int i = tid; i < a.Kmax; i += blockDim.x) {
            float v = NAN;
            if (!greedy && i < Kb) {
                const uint8_t d = ld_cg_u8(a.dec + rb + i);
                if (d == kDecAccept || d == kDecReject) {
                    const double* rc = a.Rc + (rb + i) * a.nchunks;
                    double s = 0.0;
                    for (int c = 0; c < a.nchunks; ++c)
                        s += __ldcg(rc + c);
                    v = (float)s;
                }
            }
            a.resid[(size_t)b * a.Kmax + i] = v;
        }
    }
    __syncthreads();
}

// ---------------------------------------------------------------------------
// the fused sweep kernel: one cluster per (position, sequence) row
// ---------------------------------------------------------------------------
template <typename T, int NV>
__global__ void __launch_bounds__(kMaxWarps * 32) sv_verify_kernel(const Args a)
{
    using EL = Elem<T>;
    constexpr int E = EL::E;
    constexpr int CH = 32 * NV * E;   // elements per chunk (NV 16-byte vectors per lane)

    extern __shared__ __align__(128) unsigned char dsmem[];
    __shared__ float s_wmax[kMaxWarps][2];
    __shared__ double s_wsum[kMaxWarps][2];
    __shared__ int s_widx[kMaxWarps];
    __shared__ float s_cmax[kMaxCluster][2];    // written by each cluster rank
    __shared__ double s_csum[kMaxCluster][2];
    __shared__ int s_cidx[kMaxCluster];
    __shared__ int s_skip, s_last, s_timeout;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
    const int C = a.C;
    const uint32_t rank = cluster_ctarank();
    const long long item = (long long)blockIdx.x / C;
    const int i = (int)(item / a.B);
    const int b = (int)(item - (long long)i * a.B);
    const int Kb = a.K[b];
    if (i > Kb)
        return;   // padding position of a shorter sequence: the whole cluster leaves

    const int Kmax = a.Kmax, V = a.V;
    const float Tb = a.temp[b];
    const bool greedy = (Tb == 0.0f);
    const bool is_test = i < Kb;
    const bool use_draft = is_test && !greedy;
    const size_t trow = (size_t)b * (Kmax + 1) + i;
    int x = 0;
    float u = 0.0f;
    bool in_ok = temperature_usable(Tb);
    if (is_test) {
        x = a.tok[(size_t)b * Kmax + i];
        in_ok = in_ok && x >= 0 && x < V;
        if (!greedy) {
            u = a.uni[(size_t)b * (Kmax + 1) + i];
            in_ok = in_ok && u >= 0.0f && u < 1.0f && a.drf != nullptr;
        }
    }

    // Phase A: all CTAs of the cluster have started before any DSMEM access;
    // rank 0 publishes whether a known earlier rejection makes this row moot.
    const bool may_skip = a.early_exit && i > 0;
    if (tid == 0) {
        s_timeout = 0;
        int sk = 0;
        if (may_skip && rank == 0) {
            const uint32_t m = ld_volatile_u32(a.mask + b);
            const uint32_t below = i >= 32 ? 0xffffffffu : ((1u << i) - 1u);
            sk = (m & below) != 0;
        }
        s_skip = sk;
    }
    __syncthreads();
    cluster_arrive();
    bool skip = false;
    if (may_skip) {
        cluster_wait();
        skip = ld_cluster_s32(map_to_rank(smem_addr(&s_skip), 0)) != 0;
        if (skip || !in_ok) {      // rank 0 must outlive its peers' read of s_skip
            cluster_arrive();
            cluster_wait();
        }
    } else if (!in_ok) {
        cluster_wait();
    }

    const int nck_total = a.nchunks;
    const int c0 = (int)rank * a.ncpc;
    const int nck = max(0, min(a.ncpc, nck_total - c0));
    T* s_t = reinterpret_cast<T*>(dsmem);
    T* s_d = s_t + (size_t)a.ncpc * CH;
    uint64_t* mbar = reinterpret_cast<uint64_t*>(dsmem + (size_t)2 * a.ncpc * CH * sizeof(T));
    bool issued = false;

    if (!skip && in_ok) {
        const T* tg = static_cast<const T*>(a.tgt) + trow * (size_t)V;
        const T* dg = use_draft ? static_cast<const T*>(a.drf) + ((size_t)b * Kmax + i) * (size_t)V
                                : nullptr;

        // ---- stage this CTA's chunks of the row(s) into shared memory ----
        issued = true;
        for (int lc = warp; lc < nck; lc += nw) {
            const long long e0 = (long long)(c0 + lc) * CH;
            const int n = (int)min((long long)CH, (long long)V - e0);
            const int nb = a.aligned ? ((n * (int)sizeof(T)) & ~15) / (int)sizeof(T) : 0;
            const uint32_t mb = smem_addr(&mbar[lc]);
            T* dt = s_t + (size_t)lc * CH;
            T* dd = s_d + (size_t)lc * CH;
            if (lane == 0) {
                mbar_init(mb, 1);
                fence_mbar_init();
                const uint32_t bytes = (uint32_t)nb * (uint32_t)sizeof(T);
                const uint32_t tx = bytes * (use_draft ? 2u : 1u);
                if (tx) {
                    mbar_arrive_expect_tx(mb, tx);
                    bulk_copy_g2s(smem_addr(dt), tg + e0, bytes, mb);
                    if (use_draft)
                        bulk_copy_g2s(smem_addr(dd), dg + e0, bytes, mb);
                } else {
                    mbar_arrive(mb);
                }
            }
            // ragged tail (or the whole chunk when rows are not 16-byte aligned)
            // with element loads; -inf padding up to the chunk size
            for (int j = nb + lane; j < CH; j += 32) {
                if (j < n) EL::copy(dt + j, tg + e0 + j); else EL::set_neg_inf(dt + j);
                if (use_draft) {
                    if (j < n) EL::copy(dd + j, dg + e0 + j); else EL::set_neg_inf(dd + j);
                }
            }
        }
        __syncwarp();

        // ---- pass 1: row maxima (NaN propagates) ----
        float mt = -INFINITY, md = -INFINITY;
        bool to = false;
        for (int lc = warp; lc < nck; lc += nw) {
            if (!mbar_wait_bounded(smem_addr(&mbar[lc]), 0, kWaitSpins))
                to = true;
            const uint4* vt = reinterpret_cast<const uint4*>(s_t + (size_t)lc * CH);
#pragma unroll
            for (int v = 0; v < NV; ++v) {
                float xs[E];
                EL::unpack(vt[v * 32 + lane], xs);
#pragma unroll
                for (int e = 0; e < E; ++e)
                    mt = max_nan(mt, xs[e]);
            }
            if (use_draft) {
                const uint4* vd = reinterpret_cast<const uint4*>(s_d + (size_t)lc * CH);
#pragma unroll
                for (int v = 0; v < NV; ++v) {
                    float xs[E];
                    EL::unpack(vd[v * 32 + lane], xs);
#pragma unroll
                    for (int e = 0; e < E; ++e)
                        md = max_nan(md, xs[e]);
                }
            }
        }
        if (__any_sync(kFull, to)) {
            if (lane == 0)
                s_timeout = 1;
        }
        mt = warp_max_nan(mt);
        md = warp_max_nan(md);
        if (lane == 0) {
            s_wmax[warp][0] = mt;
            s_wmax[warp][1] = md;
        }
        __syncthreads();
        if (!may_skip)
            cluster_wait();   // phase A
        if (tid < C) {
            float cm0 = -INFINITY, cm1 = -INFINITY;
            for (int w = 0; w < nw; ++w) {
                cm0 = max_nan(cm0, s_wmax[w][0]);
                cm1 = max_nan(cm1, s_wmax[w][1]);
            }
            if (s_timeout) {   // poison the row everywhere in the cluster
                cm0 = NAN;
                cm1 = NAN;
            }
            const uint32_t dst = map_to_rank(smem_addr(&s_cmax[rank][0]), (uint32_t)tid);
            st_cluster_f32(dst, cm0);
            st_cluster_f32(dst + 4, cm1);
        }
        cluster_arrive();
        cluster_wait();   // phase B
        float m_t = -INFINITY, m_d = -INFINITY;
        for (int r = 0; r < C; ++r) {
            m_t = max_nan(m_t, s_cmax[r][0]);
            m_d = max_nan(m_d, s_cmax[r][1]);
        }
        const bool ok_t = isfinite(m_t);
        const bool ok_d = !use_draft || isfinite(m_d);

        if (greedy) {
            // ---- pass 2 (greedy): lowest index holding the max ----
            int best = INT_MAX;
            if (ok_t) {
                for (int lc = warp; lc < nck; lc += nw) {
                    const uint4* vt = reinterpret_cast<const uint4*>(s_t + (size_t)lc * CH);
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
            cluster_wait();   // phase C
            int g = INT_MAX;
            for (int r = 0; r < C; ++r)
                g = min(g, s_cidx[r]);
            const bool row_ok = ok_t && g < V;
            const uint8_t d = !row_ok ? kDecInvalid
                                      : (is_test ? (x == g ? kDecAccept : kDecReject) : kDecBonus);
            if (rank == 0 && tid == 0) {
                if (is_test && d != kDecAccept)
                    atomicOr(a.mask + b, 1u << i);
                a.dec[trow] = d;
                a.argmax[trow] = row_ok ? g : -1;
                if (is_test && a.p_x) {
                    a.p_x[(size_t)b * Kmax + i] = NAN;
                    a.q_x[(size_t)b * Kmax + i] = NAN;
                }
            }
        } else {
            // ---- pass 2 (sampling): per-chunk sums of the softmax weights ----
            const float c = (float)(kLog2e / (double)Tb);
            double wst = 0.0, wsd = 0.0;
            for (int lc = warp; lc < nck; lc += nw) {
                const uint4* vt = reinterpret_cast<const uint4*>(s_t + (size_t)lc * CH);
                float acc = 0.0f;
#pragma unroll
                for (int v = 0; v < NV; ++v) {
                    float xs[E];
                    EL::unpack(vt[v * 32 + lane], xs);
#pragma unroll
                    for (int e = 0; e < E; ++e)
                        acc += weight(xs[e], m_t, c);
                }
                const double pc = warp_sum((double)acc);
                if (lane == 0)
                    a.Pc[trow * nck_total + (c0 + lc)] = pc;
                wst += pc;
                if (use_draft) {
                    const uint4* vd = reinterpret_cast<const uint4*>(s_d + (size_t)lc * CH);
                    float accd = 0.0f;
#pragma unroll
                    for (int v = 0; v < NV; ++v) {
                        float xs[E];
                        EL::unpack(vd[v * 32 + lane], xs);
#pragma unroll
                        for (int e = 0; e < E; ++e)
                            accd += weight(xs[e], m_d, c);
                    }
                    wsd += warp_sum((double)accd);
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
            cluster_wait();   // phase C
            double St = 0.0, Sd = 0.0;
            for (int r = 0; r < C; ++r) {
                St += s_csum[r][0];
                Sd += s_csum[r][1];
            }
            const bool row_ok = ok_t && ok_d && St > 0.0 && (!use_draft || Sd > 0.0);
            const float inv_st = (float)(1.0 / St);
            const float inv_sd = use_draft ? (float)(1.0 / Sd) : 0.0f;
            bool accept = false;
            float px = NAN, qx = NAN;
            if (is_test && row_ok) {
                const float et = weight(EL::load(tg + x), m_t, c);
                const float ed = weight(EL::load(dg + x), m_d, c);
                px = __fmul_rn(et, inv_st);
                qx = __fmul_rn(ed, inv_sd);
                accept = __fmul_rn(u, qx) < px;   // u < min(1, p/q) without dividing
            }
            const uint8_t d = !row_ok ? kDecInvalid
                                      : (is_test ? (accept ? kDecAccept : kDecReject) : kDecBonus);
            if (rank == 0 && tid == 0) {
                if (is_test && d != kDecAccept)
                    atomicOr(a.mask + b, 1u << i);
                a.dec[trow] = d;
                a.rowstat[trow] = make_float4(m_t, inv_st, m_d, inv_sd);
                if (is_test && a.p_x) {
                    a.p_x[(size_t)b * Kmax + i] = px;
                    a.q_x[(size_t)b * Kmax + i] = qx;
                }
            }
            // ---- pass 3: residual mass per chunk, for rows that may be drawn from ----
            if (use_draft && row_ok && (d == kDecReject || !a.early_exit)) {
                for (int lc = warp; lc < nck; lc += nw) {
                    const uint4* vt = reinterpret_cast<const uint4*>(s_t + (size_t)lc * CH);
                    const uint4* vd = reinterpret_cast<const uint4*>(s_d + (size_t)lc * CH);
                    float acc = 0.0f;
#pragma unroll
                    for (int v = 0; v < NV; ++v) {
                        float xt[E], xd[E];
                        EL::unpack(vt[v * 32 + lane], xt);
                        EL::unpack(vd[v * 32 + lane], xd);
#pragma unroll
                        for (int e = 0; e < E; ++e)
                            acc += resid_term(weight(xt[e], m_t, c), inv_st, weight(xd[e], m_d, c),
                                              inv_sd);
                    }
                    const double rc = warp_sum((double)acc);
                    if (lane == 0)
                        a.Rc[trow * nck_total + (c0 + lc)] = rc;
                }
            }
        }
    } else if (!skip && rank == 0 && tid == 0) {
        // unusable temperature, token, uniform or missing draft on this row
        if (is_test)
            atomicOr(a.mask + b, 1u << i);
        a.dec[trow] = kDecInvalid;
    }

    // A bounded wait gave up: record it, and give the copies a last bounded
    // chance to land before this CTA's shared memory is released.
    if (issued && s_timeout) {
        if (tid == 0)
            atomicOr(a.err, kErrWaitTimeout);
        for (int lc = warp; lc < nck; lc += nw)
            (void)mbar_wait_bounded(smem_addr(&mbar[lc]), 0, kWaitSpins);
    }

    // ---- arrival: the last CTA of the sequence finalises it ----
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        const int target = (Kb + 1) * C;
        const int old = atomicAdd(a.counter + b, 1);
        s_last = (old == target - 1);
    }
    __syncthreads();
    if (s_last) {
        __threadfence();
        finalize_sequence<T, NV>(a, b, Kb, Tb);
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
constexpr int kSmemPerCtaMax = 227 * 1024;   // opt-in dynamic shared memory limit
constexpr int kStaticSmemReserve = 2048;     // static __shared__ of the kernel, rounded up
constexpr int kSmemBudget = 74 * 1024;       // per-CTA target: 3 CTAs/SM at bf16, 2 at fp32

struct Geom {
    int s = 0, nv = 0, ch = 0, nchunks = 0, ncpc = 0, C = 0, nwarps = 0;
    size_t smem = 0;
};

static int elem_size(sv_dtype dt) { return dt == SV_DTYPE_BF16 ? 2 : 4; }

static int pick_nv(int V, int s)
{
    const int E = 16 / s;
    for (int nv = 8; nv > 1; nv >>= 1)
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

static size_t smem_for(int ncpc, int ch, int s)
{
    return (size_t)ncpc * (size_t)ch * (size_t)s * 2 + (size_t)ncpc * 8;
}

static int max_ncpc(int ch, int s)
{
    return (kSmemPerCtaMax - kStaticSmemReserve) / (int)smem_for(1, ch, s);
}

// Vocabulary chunks per CTA and cluster size for one launch.
static bool choose_geometry(int V, sv_dtype dt, long long items, int nsm, int override_ncpc,
                            Geom* g)
{
    const int s = elem_size(dt);
    g->s = s;
    g->nv = pick_nv(V, s);
    g->ch = 32 * g->nv * (16 / s);
    g->nchunks = (V + g->ch - 1) / g->ch;
    const int lim = max_ncpc(g->ch, s);
    int ncpc;
    if (override_ncpc > 0) {
        ncpc = override_ncpc;
    } else {
        ncpc = (int)(kSmemBudget / smem_for(1, g->ch, s));
        ncpc = max(1, min(ncpc, g->nchunks));
        if ((g->nchunks + ncpc - 1) / ncpc > kMaxCluster)
            ncpc = (g->nchunks + kMaxCluster - 1) / kMaxCluster;
        // small launches: spread each row over more CTAs (portable clusters)
        while (ncpc > 1) {
            const int half = (ncpc + 1) / 2;
            const int C2 = (g->nchunks + half - 1) / half;
            const long long ctas = items * (long long)((g->nchunks + ncpc - 1) / ncpc);
            if (C2 > 8 || ctas >= 2LL * nsm)
                break;
            ncpc = half;
        }
    }
    ncpc = min(ncpc, g->nchunks);
    int C = (g->nchunks + ncpc - 1) / ncpc;
    if (C > kMaxCluster || ncpc > lim)
        return false;
    ncpc = (g->nchunks + C - 1) / C;   // balance
    g->ncpc = ncpc;
    g->C = C;
    g->nwarps = min(ncpc, kMaxWarps);
    g->smem = smem_for(ncpc, g->ch, s);
    return true;
}

// ---- workspace layout ----
struct WsLayout {
    size_t err, counter, mask, dec, K, header_end, argmax, rowstat, Pc, Rc, total;
};

static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

static bool ws_layout(int B, int Kmax, int V, sv_dtype dt, WsLayout* L)
{
    if (B < 0 || Kmax < 0 || Kmax > SV_K_MAX || V < 1)
        return false;
    const size_t R = (size_t)B * (size_t)(Kmax + 1);
    const size_t nch = (size_t)n_chunks(V, elem_size(dt));
    size_t o = 0;
    L->err = o;      o = align256(o + 16);
    L->counter = o;  o = align256(o + (size_t)B * 4);
    L->mask = o;     o = align256(o + (size_t)B * 4);
    L->dec = o;      o = align256(o + R);
    L->K = o;        o = align256(o + (size_t)B * 4);
    L->header_end = o;
    L->argmax = o;   o = align256(o + R * 4);
    L->rowstat = o;  o = align256(o + R * 16);
    L->Pc = o;       o = align256(o + R * nch * 8);
    L->Rc = o;       o = align256(o + R * nch * 8);
    L->total = o;
    return true;
}

struct DeviceInfo {
    int nsm = 0;
    bool attrs_set[2][4] = {};
};

static std::mutex g_mu;
static DeviceInfo g_dev[64];

// Cache of cudaOccupancyMaxActiveClusters per (device, kernel, cluster size, smem).
static std::map<std::tuple<int, int, int, int, size_t>, int> g_fit;

template <typename T, int NV>
static cudaError_t prepare_kernel(int dev)
{
    auto kern = sv_verify_kernel<T, NV>;
    const int ti = sizeof(T) == 2 ? 1 : 0;
    const int ni = NV == 1 ? 0 : NV == 2 ? 1 : NV == 4 ? 2 : 3;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_dev[dev].attrs_set[ti][ni]) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             kSmemPerCtaMax - kStaticSmemReserve);
        if (e != cudaSuccess)
            return e;
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess)
            return e;
        g_dev[dev].attrs_set[ti][ni] = true;
    }
    return cudaSuccess;
}

static void fill_config(cudaLaunchConfig_t* cfg, cudaLaunchAttribute* attr, const Geom& g,
                        long long items, cudaStream_t st)
{
    *cfg = cudaLaunchConfig_t{};
    cfg->gridDim = dim3((unsigned)(items * g.C), 1, 1);
    cfg->blockDim = dim3((unsigned)(32 * g.nwarps), 1, 1);
    cfg->dynamicSmemBytes = g.smem;
    cfg->stream = st;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)g.C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg->attrs = attr;
    cfg->numAttrs = 1;
}

// How many clusters of this shape the device can hold at once (0: cannot launch).
template <typename T, int NV>
static cudaError_t cluster_capacity(const Geom& g, int dev, int* n)
{
    cudaError_t e = prepare_kernel<T, NV>(dev);
    if (e != cudaSuccess)
        return e;
    const auto key = std::make_tuple(dev, (int)sizeof(T) * 16 + NV, g.C, g.nwarps, g.smem);
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
    fill_config(&cfg, attr, g, 1, 0);
    int v = 0;
    e = cudaOccupancyMaxActiveClusters(&v, sv_verify_kernel<T, NV>, &cfg);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        v = 0;
    }
    std::lock_guard<std::mutex> lk(g_mu);
    g_fit[key] = v;
    *n = v;
    return cudaSuccess;
}

template <typename T, int NV>
static cudaError_t launch_kernel(const Args& a, const Geom& g, long long items, cudaStream_t st,
                                 int dev)
{
    cudaError_t e = prepare_kernel<T, NV>(dev);
    if (e != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[1];
    fill_config(&cfg, attr, g, items, st);
    return cudaLaunchKernelEx(&cfg, sv_verify_kernel<T, NV>, a);
}

template <typename T>
static cudaError_t launch_nv(const Args& a, const Geom& g, long long items, cudaStream_t st, int dev)
{
    switch (g.nv) {
    case 1: return launch_kernel<T, 1>(a, g, items, st, dev);
    case 2: return launch_kernel<T, 2>(a, g, items, st, dev);
    case 4: return launch_kernel<T, 4>(a, g, items, st, dev);
    default: return launch_kernel<T, 8>(a, g, items, st, dev);
    }
}

template <typename T>
static cudaError_t capacity_nv(const Geom& g, int dev, int* n)
{
    switch (g.nv) {
    case 1: return cluster_capacity<T, 1>(g, dev, n);
    case 2: return cluster_capacity<T, 2>(g, dev, n);
    case 4: return cluster_capacity<T, 4>(g, dev, n);
    default: return cluster_capacity<T, 8>(g, dev, n);
    }
}

// Pick the geometry, widening each CTA's share (smaller clusters) until the
// device can co-schedule a cluster of that shape.
static sv_status pick_launchable(int V, sv_dtype dt, long long items, int nsm, int override_ncpc,
                                 int dev, Geom* g)
{
    if (!choose_geometry(V, dt, items, nsm, override_ncpc, g))
        return SV_ERR_UNSUPPORTED;
    for (;;) {
        int n = 0;
        const cudaError_t e = dt == SV_DTYPE_BF16 ? capacity_nv<__nv_bfloat16>(*g, dev, &n)
                                                  : capacity_nv<float>(*g, dev, &n);
        if (e != cudaSuccess)
            return SV_ERR_CUDA;
        if (n > 0)
            return SV_OK;
        if (override_ncpc > 0 || g->C == 1)
            return SV_ERR_UNSUPPORTED;
        if (!choose_geometry(V, dt, items, nsm, g->ncpc + 1, g))
            return SV_ERR_UNSUPPORTED;
    }
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
    *kmax_out = kmax;
    return SV_OK;
}

static sv_status run(const Call& c, int kmax, const sv_options* opt, void* ws, size_t ws_bytes,
                     cudaStream_t stream)
{
    if (c.B == 0)
        return SV_OK;
    WsLayout L;
    if (!ws_layout(c.B, kmax, c.V, c.dtype, &L))
        return SV_ERR_INVALID_ARG;
    if (!ws || ws_bytes < L.total || ((uintptr_t)ws & 255))
        return SV_ERR_NO_MEMORY;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return SV_ERR_CUDA;
    cudaPointerAttributes pa;
    if (cudaPointerGetAttributes(&pa, c.tgt) != cudaSuccess)
        return SV_ERR_CUDA;
    if (pa.type != cudaMemoryTypeDevice && pa.type != cudaMemoryTypeManaged)
        return SV_ERR_INVALID_ARG;
    if (pa.type == cudaMemoryTypeDevice && pa.device != dev)
        return SV_ERR_INVALID_ARG;
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
    const long long items = (long long)c.B * (kmax + 1);
    Geom g;
    const sv_status gs =
        pick_launchable(c.V, c.dtype, items, nsm, opt ? opt->chunks_per_cta : 0, dev, &g);
    if (gs != SV_OK)
        return gs;
    if (items * g.C > 0x7fffffffLL)
        return SV_ERR_UNSUPPORTED;

    // Header: zeroed error word, counters, masks and decisions, then K.
    thread_local std::vector<unsigned char> hdr;
    hdr.assign(L.header_end, 0);
    memcpy(hdr.data() + L.K, c.K, (size_t)c.B * 4);
    unsigned char* base = static_cast<unsigned char*>(ws);
    if (cudaMemcpyAsync(base, hdr.data(), L.header_end, cudaMemcpyHostToDevice, stream) !=
        cudaSuccess)
        return SV_ERR_CUDA;

    const sv_diag* dg = opt ? &opt->diag : nullptr;
    const bool want_diag = dg && (dg->p_x || dg->q_x || dg->resid_mass || dg->final_row);
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
    a.ncpc = g.ncpc;
    a.C = g.C;
    a.early_exit = (want_diag || (opt && opt->verify_all)) ? 0 : 1;
    const uintptr_t al = (uintptr_t)c.tgt | (c.drf ? (uintptr_t)c.drf : 0);
    a.aligned = ((al & 15) == 0) && (((size_t)c.V * g.s) % 16 == 0);
    a.err = reinterpret_cast<uint32_t*>(base + L.err);
    a.counter = reinterpret_cast<int*>(base + L.counter);
    a.mask = reinterpret_cast<uint32_t*>(base + L.mask);
    a.dec = base + L.dec;
    a.K = reinterpret_cast<const int32_t*>(base + L.K);
    a.argmax = reinterpret_cast<int32_t*>(base + L.argmax);
    a.rowstat = reinterpret_cast<float4*>(base + L.rowstat);
    a.Pc = reinterpret_cast<double*>(base + L.Pc);
    a.Rc = reinterpret_cast<double*>(base + L.Rc);
    // p_x and q_x are written together; a lone request gets a scratch twin
    a.p_x = want_diag ? dg->p_x : nullptr;
    a.q_x = want_diag ? dg->q_x : nullptr;
    if ((a.p_x == nullptr) != (a.q_x == nullptr))
        return SV_ERR_INVALID_ARG;
    a.resid = want_diag ? dg->resid_mass : nullptr;
    a.final_row = want_diag ? dg->final_row : nullptr;

    const cudaError_t e = c.dtype == SV_DTYPE_BF16
                              ? launch_nv<__nv_bfloat16>(a, g, items, stream, dev)
                              : launch_nv<float>(a, g, items, stream, dev);
    return e == cudaSuccess ? SV_OK : SV_ERR_CUDA;
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
    const int s = sv::elem_size(dtype);
    const int ch = 32 * 8 * (16 / s);   // chunk size at large V
    return sv::kMaxCluster * sv::max_ncpc(ch, s) * ch;
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
    if (options && options->chunks_per_cta < 0)
        return SV_ERR_INVALID_ARG;
    return sv::run(c, kmax, options, workspace, workspace_bytes, stream);
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
    return (v & sv::kErrWaitTimeout) ? SV_ERR_TIMEOUT : SV_OK;
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
    if (cudaMemcpyAsync(d_tgt, h_target_logits, n_tgt, cudaMemcpyHostToDevice, stream) != cudaSuccess ||
        (has_drf && cudaMemcpyAsync(d_drf, h_draft_logits, n_drf, cudaMemcpyHostToDevice, stream) != cudaSuccess) ||
        (n_tok && cudaMemcpyAsync(d_tok, h_draft_tokens, n_tok, cudaMemcpyHostToDevice, stream) != cudaSuccess) ||
        cudaMemcpyAsync(d_uni, h_uniforms, n_uni, cudaMemcpyHostToDevice, stream) != cudaSuccess ||
        cudaMemcpyAsync(d_tmp, h_temperature, n_tmp, cudaMemcpyHostToDevice, stream) != cudaSuccess)
        return SV_ERR_CUDA;
    const sv::Call dc{d_tgt, has_drf ? d_drf : nullptr, dtype,
                      n_tok ? reinterpret_cast<const int32_t*>(d_tok) : nullptr,
                      reinterpret_cast<const float*>(d_uni), reinterpret_cast<const float*>(d_tmp),
                      B, K, V, reinterpret_cast<int32_t*>(d_otok), reinterpret_cast<int32_t*>(d_on)};
    st = sv::run(dc, kmax, nullptr, ws, ws_bytes, stream);
    if (st != SV_OK)
        return st;
    if (cudaMemcpyAsync(h_out_tokens, d_otok, n_otok, cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
        cudaMemcpyAsync(h_out_num_accepted, d_on, n_on, cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
        cudaStreamSynchronize(stream) != cudaSuccess)
        return SV_ERR_CUDA;
    return SV_OK;
}

}  // extern "C"
