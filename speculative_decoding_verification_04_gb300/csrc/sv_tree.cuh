// sv_tree.cuh -- token-tree verification: the pages' accept rule applied at
// every node of a tree of proposals (a chain of one child per node is the
// ordinary verification).
//
// A persistent cluster walks its sequences' trees (sequence c first, later
// ones claimed with an atomic ticket), each from the root.  At node v the
// cluster holds the target and draft rows after v resident in shared memory
// (the same warp ranges and bulk copies as the sweep) and tests v's children
// in index order: child c (token x) is kept iff u_c q(x) < R(x), with R = p
// at first; after a rejection R becomes normalize(max(0, R - q)) (left as it
// was if that has no mass) and the next child is tested.  A kept child is
// the next node; with none kept the token is drawn from R by inverse CDF (at
// a leaf R = p, the bonus token).  At T = 0 the child equal to the target
// argmax is kept, else the token is the argmax.
//
// Residual levels are recomputed from the resident slice, unnormalised: with
// the weights W_t = exp2(fma(l_t, c, -r_t)) and W_d (the sweep's), p = W_t / S_t
// and q = W_d / S_d, level l holds B_l = max(0, B_{l-1} - s_{l-1} W_d) with
// B_0 = W_t and s_l = sum(B_l) / S_d.  Then R_l = B_l / sum(B_l): for
// R_{l-1} = B_{l-1} / sum(B_{l-1}), max(0, R_{l-1} - q) is
// max(0, B_{l-1} - s_{l-1} W_d) / sum(B_{l-1}), and normalising it gives
// R_l.  A level without mass leaves R as it was, and then every later level
// has none either (its terms are the same), so no further level is computed.
// A pass at level L costs two exponentials and L multiply-adds per element.
// Each pass keeps per-strip partial sums of its terms for the draw, as the
// sweep's residual pass does.
#pragma once

#include "sv_sweep.cuh"

namespace sv {

constexpr int kTreeMaxNodes = 32;   // one lane per node

struct TreeArgs {
    const void* tgt;         // [B][Nmax][V]: row n, the target's logits after node n
    const void* drf;         // [B][Nmax][V]: row n, the draft's logits after node n
    const int32_t* tok;      // [B][Nmax]: node n's token (n >= 1)
    const int32_t* parent;   // [B][Nmax]: parent[n] < n, parent[0] = -1
    const float* uni;        // [B][Nmax]: uni[n] tests node n; uni[0] is the final draw
    const float* temp;       // [B]
    const int32_t* n_nodes;  // [B]
    int32_t* out_tok;        // [B][Nmax]
    int32_t* out_path;       // [B][Nmax]
    int32_t* out_len;        // [B]
    uint32_t* err;
    int* next;               // claim counter of the sequences after the first wave
    int B, Nmax, V;
    int nchunks, C, kw;
    int aligned, has_draft;
};

// The sweep's shared-memory layout (the per-level factors live in lane
// registers: lane l holds s_l), so a row's CTAs fit three to an SM as the
// sweep's do.
__host__ __device__ inline size_t tree_smem_bytes(const SweepLayout& L, int /*nw*/) { return L.total; }

// Elements 2h and 2h + 1 of a lane vector as a packed fp32 pair (lower index
// in the low lane): h = 0..3 for bf16, 0..1 for fp32.
template <typename T> struct VecPair;
template <> struct VecPair<__nv_bfloat16> {
    __device__ static __forceinline__ uint64_t get(const uint4& q, int h)
    {
        return Lane<__nv_bfloat16, 1>::pair(h == 0 ? q.x : h == 1 ? q.y : h == 2 ? q.z : q.w);
    }
};
template <> struct VecPair<float> {
    __device__ static __forceinline__ uint64_t get(const uint4& q, int h)
    {
        return h == 0 ? f2_pack(__uint_as_float(q.x), __uint_as_float(q.y))
                      : f2_pack(__uint_as_float(q.z), __uint_as_float(q.w));
    }
};

// The level-L terms B_L of one 16-byte vector pair (E elements, lane order),
// elements in packed pairs: W_t and W_d by a packed fma and two ex2 each,
// then per level one packed multiply-add and a clamp at 0.  LC = min(L, 3)
// (a compile-time level class); n0, n1 hold -s_0 and -s_1 packed, levels
// from 2 on shuffle s_l from lane l of `sig`.  Every element's value is the
// same rounding sequence whichever way the factors arrive.
template <typename T, int NV, int LC>
__device__ __forceinline__ void level_terms_vec(const uint4& tv, const uint4& dv, uint64_t Cc, uint64_t NT,
                                                uint64_t ND, int L, uint64_t n0, uint64_t n1, float sig,
                                                float (&out)[Elem<T>::E])
{
    constexpr int E = Elem<T>::E;
#pragma unroll
    for (int h = 0; h < E / 2; ++h) {
        float a0, a1;
        f2_unpack(f2_fma(VecPair<T>::get(tv, h), Cc, NT), a0, a1);
        uint64_t b = f2_pack(ex2_approx(a0), ex2_approx(a1));
        if (LC > 0) {
            f2_unpack(f2_fma(VecPair<T>::get(dv, h), Cc, ND), a0, a1);
            const uint64_t wd = f2_pack(ex2_approx(a0), ex2_approx(a1));
            f2_unpack(f2_fma(n0, wd, b), a0, a1);
            b = f2_pack(fmaxf(a0, 0.0f), fmaxf(a1, 0.0f));
            if (LC > 1) {
                f2_unpack(f2_fma(n1, wd, b), a0, a1);
                b = f2_pack(fmaxf(a0, 0.0f), fmaxf(a1, 0.0f));
            }
            if (LC > 2) {
                for (int l = 2; l < L; ++l) {
                    const float s = __shfl_sync(kFull, sig, l);
                    f2_unpack(f2_fma(f2_pack(-s, -s), wd, b), a0, a1);
                    b = f2_pack(fmaxf(a0, 0.0f), fmaxf(a1, 0.0f));
                }
            }
        }
        f2_unpack(b, out[2 * h], out[2 * h + 1]);
    }
}

// -s_0 and -s_1, packed, for level_terms_vec (every lane).
__device__ __forceinline__ void level_factors(float sig, uint64_t& n0, uint64_t& n1)
{
    const float s0 = __shfl_sync(kFull, sig, 0), s1 = __shfl_sync(kFull, sig, 1);
    n0 = f2_pack(-s0, -s0);
    n1 = f2_pack(-s1, -s1);
}

// B_k(x) for the proposal's weights W_t(x), W_d(x) (the same steps as
// level_terms_vec, one lane of them).
__device__ __forceinline__ float level_value(float wt, float wd, int k, float sig)
{
    float b = wt;
    for (int l = 0; l < k; ++l)
        b = fmaxf(__fmaf_rn(-__shfl_sync(kFull, sig, l), wd, b), 0.0f);
    return b;
}

// One pass over this warp's slice at level L (whole warp): per-strip partial
// sums of the level's terms into `stats` ([kw][NV][4], as the sweep's
// residual pass), and the warp's total (compensated); terms as in
// level_terms_vec.
template <typename T, int NV, int LC>
__device__ float level_pass_lc(const T* slot_t, const T* slot_d, int kwm, int lane, float c, float rt, float rd,
                               int L, float sig, float* stats)
{
    constexpr int E = Elem<T>::E;
    constexpr int CH = 32 * NV * E;
    const uint64_t Cc = f2_pack(c, c), NT = f2_pack(-rt, -rt), ND = f2_pack(-rd, -rd);
    uint64_t n0, n1;
    level_factors(sig, n0, n1);
    float acc = 0.0f, cmp = 0.0f;
#pragma unroll 1
    for (int j = 0; j < kwm; ++j) {
        uint4 tv[NV], dv[NV];
        load_chunk<T, NV>(slot_t + (size_t)j * CH, lane, tv);
        load_chunk<T, NV>(slot_d + (size_t)j * CH, lane, dv);
        float sv[NV];
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            float tm[E];
            level_terms_vec<T, NV, LC>(tv[k], dv[k], Cc, NT, ND, L, n0, n1, sig, tm);
            float sk = 0.0f;
#pragma unroll
            for (int e = 0; e < E; ++e)
                sk += tm[e];
            sv[k] = sk;
        }
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
    return sum_or_special(acc + cmp);
}

template <typename T, int NV>
__device__ float level_pass(const T* slot_t, const T* slot_d, int kwm, int lane, float c, float rt, float rd,
                            int L, float sig, float* stats)
{
    switch (L) {
    case 0: return level_pass_lc<T, NV, 0>(slot_t, slot_d, kwm, lane, c, rt, rd, L, sig, stats);
    case 1: return level_pass_lc<T, NV, 1>(slot_t, slot_d, kwm, lane, c, rt, rd, L, sig, stats);
    case 2: return level_pass_lc<T, NV, 2>(slot_t, slot_d, kwm, lane, c, rt, rd, L, sig, stats);
    default: return level_pass_lc<T, NV, 3>(slot_t, slot_d, kwm, lane, c, rt, rd, L, sig, stats);
    }
}

// The element of one strip that holds the point tc of the level-L
// distribution (one warp; tv / dv: each lane's vector of the strip): lane
// sums, a compensated scan, the lane, then the element, the terms computed
// exactly as in level_pass (level_terms_vec).  Returns lane * E + e, or -1 if the strip has no
// mass; beyond the strip's mass (rounding) the last element with mass.
template <typename T, int NV>
__device__ int pick_level(const uint4& tv, const uint4& dv, float c, float rt, float rd, int L, float sig,
                          float tc, bool beyond, int lane)
{
    constexpr int E = Elem<T>::E;
    float tm[E];
    float ls = 0.0f;
    int lastpos = -1;
    uint64_t n0, n1;
    level_factors(sig, n0, n1);
    const uint64_t Cc = f2_pack(c, c), NT = f2_pack(-rt, -rt), ND = f2_pack(-rd, -rd);
    switch (L) {
    case 0: level_terms_vec<T, NV, 0>(tv, dv, Cc, NT, ND, L, n0, n1, sig, tm); break;
    case 1: level_terms_vec<T, NV, 1>(tv, dv, Cc, NT, ND, L, n0, n1, sig, tm); break;
    case 2: level_terms_vec<T, NV, 2>(tv, dv, Cc, NT, ND, L, n0, n1, sig, tm); break;
    default: level_terms_vec<T, NV, 3>(tv, dv, Cc, NT, ND, L, n0, n1, sig, tm); break;
    }
#pragma unroll
    for (int e = 0; e < E; ++e) {
        ls += tm[e];
        if (tm[e] > 0.0f)
            lastpos = lane * E + e;
    }
    int cand = -1;
    if (!beyond) {
        float ss, sc;
        warp_incl_scan_comp(ls, lane, ss, sc);
        const unsigned hit = __ballot_sync(kFull, ls > 0.0f && tc < ss + sc);
        if (hit) {
            const int src = __ffs(hit) - 1;
            const float tl = tc - ((ss - ls) + sc);
            int ce = -1, lp = -1;
            float cum = 0.0f;
#pragma unroll
            for (int e = 0; e < E; ++e) {
                cum += tm[e];
                if (tm[e] > 0.0f) {
                    lp = e;
                    if (ce < 0 && tl < cum)
                        ce = e;
                }
            }
            ce = ce >= 0 ? ce : lp;
            cand = __shfl_sync(kFull, lane * E + ce, src);
        }
    }
    if (cand < 0)
        cand = __reduce_max_sync(kFull, lastpos);
    return cand;
}

template <typename T, int NV>
__global__ void __maxnreg__(kMaxRegs) sv_tree_kernel(const TreeArgs a)
{
    using EL = Elem<T>;
    using LN = Lane<T, NV>;
    constexpr int E = EL::E;
    constexpr int CH = 32 * NV * E;
    extern __shared__ __align__(128) unsigned char dsm[];

    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int nw = (int)(blockDim.x >> 5);
    const int C = a.C, V = a.V, Nmax = a.Nmax, KW = a.kw;
    const int P = C * nw;
    const uint32_t rank = cluster_ctarank();
    const int g = (int)rank * nw + w;
    const int c_lo = range_lo(g, a.nchunks, P);
    const int kwm = range_lo(g + 1, a.nchunks, P) - c_lo;
    const int e0 = c_lo * CH;
    const int n_el = max(0, min(e0 + kwm * CH, V) - e0);
    const SweepLayout L = sweep_layout(nw, cta_chunks(a.nchunks, C), KW, CH * (int)sizeof(T), P);
    const size_t off = (size_t)(c_lo - range_lo((int)rank * nw, a.nchunks, P)) * CH;
    T* slot_t = reinterpret_cast<T*>(dsm) + off;
    T* slot_d = reinterpret_cast<T*>(dsm + L.region_bytes) + off;
    const uint32_t bar = smem_addr(dsm + L.bars + 8 * (size_t)w);
    uint64_t* xbar = reinterpret_cast<uint64_t*>(dsm + L.xbar);
    uint64_t* xbar2 = reinterpret_cast<uint64_t*>(dsm + L.xbar2);
    const uint32_t xbarc = smem_addr(dsm + L.xbarc);
    const int* first_seq = reinterpret_cast<const int*>(dsm + L.first);
    float4* xbuf = reinterpret_cast<float4*>(dsm + L.xbuf);
    float2* xbuf2 = reinterpret_cast<float2*>(dsm + L.xbuf2);
    int2* xclaim = reinterpret_cast<int2*>(dsm + L.xclaim);   // [2]: the next tree, sent with a row exchange
    float* stats = reinterpret_cast<float*>(dsm + L.stats) + (size_t)w * KW * 16;

    if (lane == 0) {
        mbar_init(bar, 1);
        if (w == 0) {
            mbar_init(smem_addr(&xbar[0]), 1);
            mbar_init(smem_addr(&xbar[1]), 1);
            mbar_init(smem_addr(&xbar2[0]), 1);
            mbar_init(smem_addr(&xbar2[1]), 1);
            mbar_init(xbarc, 1);
        }
        fence_mbar_init();
    }
    for (int j = n_el + lane; j < kwm * CH; j += 32) {
        EL::set_neg_inf(slot_t + j);
        EL::set_neg_inf(slot_d + j);
    }
    __syncthreads();
    cluster_arrive();
    cluster_wait();

    const T* tgt = static_cast<const T*>(a.tgt);
    const T* drf = static_cast<const T*>(a.drf);
    const bool writer = rank == 0 && w == 0;
    const int n_clusters = (int)(gridDim.x / (unsigned)C);
    const int cid = (int)(blockIdx.x / (unsigned)C);

    uint32_t uses = 0, kx = 0, k2 = 0, kc = 0;
    uint32_t kx_claim = 0;   // row exchanges run when the last claim was read
    // While two waves of trees remain, the next tree is claimed a tree
    // ahead: rank 0's writer takes a ticket when a tree starts and sends it
    // with the tree's first row exchange, so the claim's round trip and the
    // next root rows' reads overlap the walk (-2: not known yet; -1: none
    // left).  Nearer the end it is claimed when the tree ends.
    int next_tree = -2;
    float next_T = 0.0f;   // its temperature (its draft row is prefetched only if > 0)
    int ticket = -1;       // the writer's ticket for the next tree
    const int nb_pf = a.aligned ? ((n_el * (int)sizeof(T)) & ~15) / (int)sizeof(T) : 0;
    float sig = 0.0f;        // lane l: s_l = sum(B_l) / S_d of the node's residual levels
    bool pending = false, xbroken = false;
    // the current sequence (lane n: node n), set when it starts
    int b = 0, N = 0, par = -2, tokn = 0;
    int path_l = -1;   // lane j: the j-th kept node
    float Tb = 0.0f, un = 0.0f, c = 0.0f;
    bool bad = false, greedy = false, done = false;

    // outputs of the sequence (whole warp; one warp calls it): the kept
    // nodes and their tokens, then `token`; token < 0 marks unusable input
    auto write_out = [&](int len, int token) {
        const bool ok = token >= 0;
        const int ptok = __shfl_sync(kFull, tokn, path_l & 31);
        if (lane < Nmax) {
            a.out_path[(size_t)b * Nmax + lane] = (ok && lane < len) ? path_l : -1;
            a.out_tok[(size_t)b * Nmax + lane] = !ok ? -1 : (lane < len ? ptok : (lane == len ? token : -1));
        }
        if (lane == 0)
            a.out_len[b] = ok ? len : -1;
    };
    // the copies of this warp's range of row `row` (and of the draft row)
    auto issue = [&](size_t row, bool with_d) {
        if (n_el <= 0)
            return;
        const T* tr = tgt + row * (size_t)V + e0;
        const T* dr = with_d ? drf + row * (size_t)V + e0 : nullptr;
        const int nb = a.aligned ? ((n_el * (int)sizeof(T)) & ~15) / (int)sizeof(T) : 0;
        if (lane == 0) {
            const uint32_t bytes = (uint32_t)nb * (uint32_t)sizeof(T);
            const uint32_t tx = bytes * (with_d ? 2u : 1u);
            if (tx) {
                fence_proxy_async();
                mbar_arrive_expect_tx(bar, tx);
                bulk_copy_g2s(smem_addr(slot_t), tr, bytes, bar);
                if (with_d)
                    bulk_copy_g2s(smem_addr(slot_d), dr, bytes, bar);
            } else {
                mbar_arrive(bar);
            }
        }
        for (int j = nb + lane; j < n_el; j += 32) {
            EL::copy(slot_t + j, tr + j);
            if (with_d)
                EL::copy(slot_d + j, dr + j);
        }
        pending = true;
    };
    // a float4 per warp to every CTA; every warp returns the P partials
    // (lane j: warp j's).  With `claim`, rank 0's writer also sends the next
    // tree (`claimed`, its lane 0) and every warp reads it into next_tree.
    auto exchange4 = [&](float4 part, bool claim, int claimed, float claimedT) -> float4 {
        const int p = (int)(kx & 1);
        const uint32_t par4 = (kx >> 1) & 1u;
        ++kx;
        if (w == 0 && lane == 0)
            mbar_arrive_expect_tx(smem_addr(&xbar[p]), (uint32_t)P * 16u + (claim ? 8u : 0u));
        const int cb = __shfl_sync(kFull, claimed, 0);
        const float cT = __shfl_sync(kFull, claimedT, 0);
        if (lane < C) {
            const uint32_t rb = map_to_rank(smem_addr(&xbar[p]), (uint32_t)lane);
            st_async_v4(map_to_rank(smem_addr(&xbuf[p * P + g]), (uint32_t)lane), part, rb);
            if (writer && claim)
                st_async_v2(map_to_rank(smem_addr(&xclaim[p]), (uint32_t)lane),
                            make_float2(__int_as_float(cb), cT), rb);
        }
        if (!mbar_wait_bounded(smem_addr(&xbar[p]), par4, kWaitSpins))
            xbroken = true;
        if (claim && !xbroken) {
            next_tree = xclaim[p].x;
            next_T = __int_as_float(xclaim[p].y);
        }
        return lane < P ? xbuf[p * P + lane] : make_float4(-INFINITY, __int_as_float(INT_MAX), -INFINITY, 0.0f);
    };
    auto exchange2 = [&](float v) -> float {
        const int p = (int)(k2 & 1);
        const uint32_t par2 = (k2 >> 1) & 1u;
        ++k2;
        if (w == 0 && lane == 0)
            mbar_arrive_expect_tx(smem_addr(&xbar2[p]), (uint32_t)P * 8u);
        if (lane < C)
            st_async_v2(map_to_rank(smem_addr(&xbuf2[p * P + g]), (uint32_t)lane), make_float2(v, 0.0f),
                        map_to_rank(smem_addr(&xbar2[p]), (uint32_t)lane));
        if (!mbar_wait_bounded(smem_addr(&xbar2[p]), par2, kWaitSpins))
            xbroken = true;
        return lane < P ? xbuf2[p * P + lane].x : 0.0f;
    };

    // ---- sequence cid, then claimed ones ----
    for (int bb = cid; bb >= 0 && bb < a.B && !xbroken;) {
    b = bb;
    N = __ldg(a.n_nodes + b);
    Tb = __ldg(a.temp + b);
    par = -2;
    tokn = 0;
    un = 0.0f;
    if (lane < Nmax) {
        par = __ldg(a.parent + (size_t)b * Nmax + lane);
        tokn = __ldg(a.tok + (size_t)b * Nmax + lane);
        un = __ldg(a.uni + (size_t)b * Nmax + lane);
    }
    const bool tree_ok = N >= 1 && N <= Nmax &&
                         !__any_sync(kFull, lane >= 1 && lane < N && (par < 0 || par >= lane));
    bad = !tree_ok || !temperature_usable(Tb);
    greedy = Tb == 0.0f;
    c = (!bad && !greedy) ? log2e_over(Tb) : 0.0f;
    path_l = -1;
    done = false;
    next_tree = -2;
    // claimed ahead (tree ids are tickets); else when this tree ends, so
    // that the last trees go to the clusters that are free first
    const bool ahead = (long long)b + 2LL * n_clusters < (long long)a.B;
    ticket = -1;
    if (ahead && writer && lane == 0)
        ticket = atomicAdd(a.next, 1) + n_clusters;

    // ---- the walk: one node per step ----
    int v = 0, len = 0;
    for (int step = 0; !bad && step < N; ++step) {
        const unsigned kids = __ballot_sync(kFull, lane > v && lane < N && par == v);
        const bool with_d = !greedy && kids != 0;
        if (with_d && !a.has_draft) {
            bad = true;
            break;
        }
        const size_t row = (size_t)b * Nmax + v;
        issue(row, with_d);
        // each child's lane loads the two logits at its token now; the tests
        // read them after the pass
        uint32_t klt = 0u, kld = 0u;
        if (with_d && ((kids >> lane) & 1u) && tokn >= 0 && tokn < V) {
            klt = EL::load_raw(tgt + row * (size_t)V + tokn);
            kld = EL::load_raw(drf + row * (size_t)V + tokn);
        }
        bool have = false;
        if (pending) {
            const bool okw = mbar_wait_bounded(bar, uses & 1u, kWaitSpins);
            have = !__any_sync(kFull, !okw);
            if (have) {
                pending = false;
                ++uses;
            } else {
                xbroken = true;
            }
            __syncwarp();
        }
        if (__any_sync(kFull, xbroken))
            break;

        // the next tree (claimed ahead): rank 0's writer sends it (and its
        // temperature) with this tree's first row exchange; its ticket was
        // taken at the start
        const bool claim_now = ahead && next_tree == -2;
        int cl = -1;
        float clT = 0.0f;
        if (claim_now && writer && lane == 0) {
            cl = (ticket >= 0 && ticket < a.B) ? ticket : -1;
            clT = cl >= 0 ? __ldg(a.temp + cl) : 0.0f;
        }

        // ---- pass: the argmax; at a sampling node with children the sums of
        // the target and draft weights against the first child's logits (no
        // max pass, and every warp's partials share the reference and add;
        // weighed again against the maxima if a weight overflows); at a leaf
        // the maximum, then per-strip sums of p's weights against it, which
        // the draw uses as they are ----
        const int c1 = kids ? __ffs(kids) - 1 : 0;
        const float ref_t = EL::widen(__shfl_sync(kFull, klt, c1));
        const float ref_d = EL::widen(__shfl_sync(kFull, kld, c1));
        const int x1 = __shfl_sync(kFull, tokn, c1);
        bool refmode = !greedy && with_d && x1 >= 0 && x1 < V && isfinite(ref_t) && isfinite(ref_d);
        const bool leaf = !greedy && !with_d;
        float4 xv;
        for (int attempt = 0; attempt < 2; ++attempt) {
        float4 part = make_float4(-INFINITY, __int_as_float(INT_MAX), -INFINITY, 0.0f);
        if (greedy) {
            // the lane's maximum and the first chunk holding it (selects, no
            // branch), then one search of that chunk for the lowest element
            float gm = -INFINITY;
            int gi = INT_MAX, gj = -1;
#pragma unroll 1
            for (int j = 0; have && j < kwm; ++j) {
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
            const float m = warp_max_nan(gm);
            part = make_float4(m, __int_as_float(__reduce_min_sync(kFull, gm == m ? gi : INT_MAX)), -INFINITY,
                               0.0f);
        } else if (refmode) {
            float st = 0.0f, sd = 0.0f;
#pragma unroll 1
            for (int j = 0; have && j < kwm; ++j) {
                uint4 vv[NV];
                load_chunk<T, NV>(slot_t + (size_t)j * CH, lane, vv);
                st += LN::exp_sum(vv, ref_t, c);
                load_chunk<T, NV>(slot_d + (size_t)j * CH, lane, vv);
                sd += LN::exp_sum(vv, ref_d, c);
            }
            sum_or_special2(st, sd);   // an overflowed weight gives +inf
            part = make_float4(ref_t, st, ref_d, sd);
        } else if (leaf) {
            float lm = -INFINITY, acc = 0.0f, cmp = 0.0f;
#pragma unroll 1
            for (int j = 0; have && j < kwm; ++j) {
                uint4 tv[NV];
                load_chunk<T, NV>(slot_t + (size_t)j * CH, lane, tv);
                lm = max_nan(lm, LN::max(tv));
            }
            const float mm = warp_max_nan(lm);
            const float mu = mm == -INFINITY ? 0.0f : mm;
#pragma unroll 1
            for (int j = 0; have && j < kwm; ++j) {
                uint4 tv[NV];
                load_chunk<T, NV>(slot_t + (size_t)j * CH, lane, tv);
                float sv[NV];
                LN::exp_strips(tv, mu, c, sv);
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
            part = make_float4(mm, sum_or_special(acc + cmp), -INFINITY, 0.0f);
        } else {
            float mt = -INFINITY, st = 0.0f, md = -INFINITY, sd = 0.0f;
#pragma unroll 1
            for (int j = 0; have && j < kwm; ++j) {
                uint4 tv[NV];
                load_chunk<T, NV>(slot_t + (size_t)j * CH, lane, tv);
                const float nt = max_nan(mt, LN::max(tv));
                if (nt != mt) {
                    st = mt == -INFINITY ? 0.0f : st * weight(mt, nt, c);
                    mt = nt;
                }
                st += LN::exp_sum(tv, mt == -INFINITY ? 0.0f : mt, c);
                if (with_d) {
                    uint4 dv[NV];
                    load_chunk<T, NV>(slot_d + (size_t)j * CH, lane, dv);
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
        }
        xv = exchange4(part, claim_now && attempt == 0, cl, clT);
        if (claim_now && attempt == 0 && !xbroken) {
            // this warp's range of the next tree's root rows, into L2
            if (next_tree >= 0 && lane == 0 && nb_pf > 0) {
                const size_t nrow = (size_t)next_tree * Nmax;
                bulk_prefetch_l2(tgt + nrow * (size_t)V + e0, (uint32_t)nb_pf * (uint32_t)sizeof(T));
                if (a.has_draft && next_T != 0.0f)
                    bulk_prefetch_l2(drf + nrow * (size_t)V + e0, (uint32_t)nb_pf * (uint32_t)sizeof(T));
            }
        }
        if (__any_sync(kFull, xbroken))
            break;
        if (refmode) {
            const bool any_inf = __any_sync(kFull, lane < P && (isinf(xv.y) || isinf(xv.w)));
            const bool any_nan = __any_sync(kFull, lane < P && (isnan(xv.x) || isnan(xv.y) || isnan(xv.z) ||
                                                               isnan(xv.w)));
            if (any_inf && !any_nan) {   // the same slice again, weighed against the maxima
                refmode = false;
                continue;
            }
        }
        break;
        }
        if (__any_sync(kFull, xbroken))
            break;

        if (greedy) {
            const float m_t = warp_max_nan(xv.x);
            const int gtok = __reduce_min_sync(kFull, (lane < P && xv.x == m_t) ? __float_as_int(xv.y) : INT_MAX);
            if (!isfinite(m_t) || gtok < 0 || gtok >= V) {
                bad = true;
                break;
            }
            // children are tested in order up to the first that holds the argmax
            const unsigned hit = __ballot_sync(kFull, ((kids >> lane) & 1u) && tokn == gtok);
            const int first = hit ? __ffs(hit) - 1 : 32;
            if (__any_sync(kFull, ((kids >> lane) & 1u) && lane < first && (tokn < 0 || tokn >= V))) {
                bad = true;
                break;
            }
            if (hit) {
                const int cn = __ffs(hit) - 1;
                if (lane == len)
                    path_l = cn;
                ++len;
                v = cn;
                continue;
            }
            if (writer)
                write_out(len, gtok);
            done = true;
            break;
        }

        // ---- sampling: p and q of the row, then the children in order ----
        if (__any_sync(kFull, lane < P && (isnan(xv.x) || isnan(xv.y) || isnan(xv.z) || isnan(xv.w)))) {
            bad = true;
            break;
        }
        float m_t, S_t, m_d, S_d;
        if (refmode) {   // every warp weighed against the first child's logits
            m_t = ref_t;
            m_d = ref_d;
            S_t = lane < P ? xv.y : 0.0f;
            S_d = lane < P ? xv.w : 0.0f;
            warp_sum_comp2(S_t, S_d);
        } else {
            combine_ms2(xv.x, xv.y, xv.z, xv.w, c, m_t, S_t, m_d, S_d);
        }
        if (!(isfinite(m_t) && S_t > 0.0f && isfinite(S_t)) ||
            (with_d && !(isfinite(m_d) && S_d > 0.0f && isfinite(S_d)))) {
            bad = true;
            break;
        }
        const float ist = __frcp_rn(S_t), isd = with_d ? __frcp_rn(S_d) : 0.0f;
        const float rt = ref_of(m_t, c), rd = with_d ? ref_of(m_d, c) : 0.0f;
        int k = 0;              // residual levels applied (each with mass): R = B_k / sum(B_k)
        bool dead = false;      // a level came out without mass: R stays as it is
        float ib = ist;         // 1 / sum(B_k)
        if (lane == 0)
            sig = __fmul_rn(S_t, isd);   // s_0 = sum(B_0) / S_d
        int stats_level = -1;   // the level whose terms the strip partials hold
        float wmass = 0.0f;     // lane j: warp j's total of the stats level
        if (leaf) {   // the pass kept p's strips (against each warp's maximum)
            stats_level = 0;
            wmass = (lane < P && xv.x != -INFINITY) ? __fmul_rn(xv.y, weight(xv.x, m_t, c)) : 0.0f;   // B_0 units
        }
        bool moved = false;
        // each child's weights W_t(x), W_d(x) and q(x) in its own lane, and
        // which children are usable (token in range, uniform in [0, 1))
        const bool is_kid = (kids >> lane) & 1u;
        const float wt_l = is_kid ? weight_r(EL::widen(klt), rt, c) : 0.0f;
        const float wd_l = is_kid ? weight_r(EL::widen(kld), rd, c) : 0.0f;
        const float qx_l = __fmul_rn(wd_l, isd);
        const unsigned kid_ok =
            __ballot_sync(kFull, is_kid && tokn >= 0 && tokn < V && un >= 0.0f && un < 1.0f);
        unsigned rest = kids;
        while (rest) {
            const int cn = __ffs(rest) - 1;
            rest &= rest - 1;
            if (!((kid_ok >> cn) & 1u)) {
                bad = true;
                break;
            }
            // every child lane tests itself against R_k; child cn's result counts
            const float r_l = __fmul_rn(level_value(wt_l, wd_l, k, sig), ib);   // R_k(x)
            const bool keep_l = qx_l > 0.0f ? __fmul_rn(un, qx_l) < r_l : r_l > 0.0f;
            const bool keep = (__ballot_sync(kFull, keep_l) >> cn) & 1u;
            if (keep) {
                if (lane == len)
                    path_l = cn;
                ++len;
                v = cn;
                moved = true;
                break;
            }
            if (dead)
                continue;   // R unchanged: the next child is tested against it
            // the next residual level, from the resident slice
            const float tot =
                have ? level_pass<T, NV>(slot_t, slot_d, kwm, lane, c, rt, rd, k + 1, sig, stats) : 0.0f;
            wmass = exchange2(tot);
            if (__any_sync(kFull, xbroken))
                break;
            const float S = warp_sum_comp(wmass);
            if (!(S >= 0.0f && isfinite(S))) {
                bad = true;
                break;
            }
            stats_level = k + 1;
            if (S > 0.0f) {
                ++k;
                if (lane == k)
                    sig = __fmul_rn(S, isd);
                ib = __frcp_rn(S);
            } else {
                dead = true;
            }
        }
        const int draw_level = k;   // the last level with mass (0: p itself)
        if (bad || __any_sync(kFull, xbroken))
            break;
        if (moved)
            continue;

        // ---- no child kept: the token from R (at a leaf R = p) ----
        const float u0 = __shfl_sync(kFull, un, 0);
        if (!(u0 >= 0.0f && u0 < 1.0f)) {
            bad = true;
            break;
        }
        if (stats_level != draw_level) {   // strips of the level drawn from
            const float tot =
                have ? level_pass<T, NV>(slot_t, slot_d, kwm, lane, c, rt, rd, draw_level, sig, stats)
                     : 0.0f;
            wmass = exchange2(tot);
            if (__any_sync(kFull, xbroken))
                break;
        }
        float t = 0.0f;
        bool beyond = false;
        int owner = -1;
        {
            float sw, cw;
            warp_incl_scan_comp(wmass, lane, sw, cw);
            const float S = __shfl_sync(kFull, sw, 31) + __shfl_sync(kFull, cw, 31);
            if (S > 0.0f && isfinite(S)) {
                t = u0 * S;
                const unsigned hit = __ballot_sync(kFull, lane < P && wmass > 0.0f && t < sw + cw);
                if (hit) {
                    owner = __ffs(hit) - 1;
                    const float os = __shfl_sync(kFull, sw, owner);
                    const float oc = __shfl_sync(kFull, cw, owner);
                    const float ow = __shfl_sync(kFull, wmass, owner);
                    t = t - ((os - ow) + oc);
                } else {
                    const unsigned posm = __ballot_sync(kFull, lane < P && wmass > 0.0f);
                    owner = posm ? 31 - __clz(posm) : -1;
                    beyond = true;
                }
            }
        }
        if (owner < 0) {
            if (writer)
                write_out(len, -1);
        } else if (owner == g) {
            // a leaf's strips were summed against this warp's own maximum:
            // rescaled to B_0 = W_t (against the row's maximum)
            const float own_m = __shfl_sync(kFull, xv.x, g & 31);
            const float sscale = (leaf && draw_level == 0)
                                     ? (own_m == -INFINITY ? 0.0f : weight(own_m, m_t, c))
                                     : 1.0f;
            auto strip_mass = [&](int q) -> float {
                const float4 m4 = *reinterpret_cast<const float4*>(stats + (size_t)q * 4);
                return ((m4.x + m4.y) + (m4.z + m4.w)) * sscale;
            };
            float tc = t;
            int token = -1;
            const int js = select_cdf(kwm * NV, strip_mass, tc, beyond, lane);
            if (js >= 0) {
                const int jc = js / NV, ks = js % NV;
                const uint4 t4 = reinterpret_cast<const uint4*>(slot_t + (size_t)jc * CH)[ks * 32 + lane];
                const uint4 d4 = reinterpret_cast<const uint4*>(slot_d + (size_t)jc * CH)[ks * 32 + lane];
                const int ce = pick_level<T, NV>(t4, d4, c, rt, rd, draw_level, sig, tc, beyond, lane);
                if (ce >= 0)
                    token = e0 + jc * CH + ks * 32 * E + ce;
            }
            write_out(len, (token >= 0 && token < V) ? token : -1);
        }
        done = true;
        break;
    }
    if (!done && writer)
        write_out(len, -1);
    if (__any_sync(kFull, xbroken))
        break;
    // the next sequence: rank 0's writer takes a ticket and sends it to every
    // CTA (st.async onto each CTA's claim mbarrier, bounded wait).  Every
    // warp must have read the previous claim first: a row exchange since then
    // shows it; a sequence rejected before its walk (no exchange) waits at a
    // cluster barrier instead (uniform: it follows from the sequence's data).
    if (next_tree != -2) {   // claimed with the tree's first row exchange
        bb = next_tree;
    } else {
        if (kc > 0 && kx == kx_claim) {
            cluster_arrive();
            cluster_wait();
        }
        if (w == 0 && lane == 0)
            mbar_arrive_expect_tx(xbarc, 8u);
        int nb = -1;
        if (writer && lane == 0)
            nb = ahead ? ticket : atomicAdd(a.next, 1) + n_clusters;
        nb = __shfl_sync(kFull, nb, 0);
        if (writer && lane < C)
            st_async_v2(map_to_rank(smem_addr(first_seq), (uint32_t)lane),
                        make_float2(__int_as_float(nb), 0.0f), map_to_rank(xbarc, (uint32_t)lane));
        if (!mbar_wait_bounded(xbarc, kc & 1u, kWaitSpins))
            xbroken = true;
        ++kc;
        if (__any_sync(kFull, xbroken))
            break;
        bb = *first_seq;
        kx_claim = kx;
    }
    }

    // ---- wind-down: a copy still in flight (only after a timeout), then
    // leave together (no CTA exits while a peer may still address it) ----
    if (xbroken) {
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
