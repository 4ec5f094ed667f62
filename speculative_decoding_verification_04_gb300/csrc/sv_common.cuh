// sv_common.cuh -- shared device definitions of libspecverify: kernel
// arguments, element access, the fixed-rounding softmax weight, warp
// reductions and the per-row decision codes.
#pragma once

#include <cuda_bf16.h>
#include <float.h>
#include <limits.h>
#include <math.h>
#include <stdint.h>

#include "sv_ptx.cuh"

namespace sv {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kMaxWarps = 8;
// Registers per thread of the sweep: an SM sub-partition's 16K registers
// then hold three warps (nine to twelve per SM, the geometries the resident
// row slices lead to).
constexpr int kMaxRegs = 168;
constexpr int kMaxCluster = 16;
constexpr uint32_t kWaitSpins = 1u << 22;   // bounded mbarrier polls (a few seconds)
// Clusters whose first sequence comes with the launch arguments (cluster c
// starts with ticket c; the tickets after the first wave are claimed).
constexpr int kFirstUnits = 256;
// Decision of one row.
enum : int {
    kDecAccept = 1,
    kDecReject = 2,
    kDecInvalid = 3,   // unusable input on this row
    kDecBonus = 4,     // position K_b evaluated and usable
    kDecRedo = 5       // weigh the row again against its maxima
};

// bit 0: a bounded wait gave up; bit 1: a sequence the caller's temperature
// hint called greedy has a nonzero device temperature (its outputs are -1)
enum : uint32_t { kErrWaitTimeout = 1u, kErrHint = 2u };

struct Args {
    const void* tgt;
    const void* drf;
    const int32_t* tok;
    const float* uni;
    const float* temp;
    int32_t* out_tok;
    int32_t* out_n;
    int B, Kmax, V;
    int nchunks;           // vocabulary chunks per row
    int C;                 // CTAs per cluster (one row at a time per cluster)
    int kw;                // chunks per warp (a contiguous range)
    int early_exit, aligned;
    // Which optional buffers were supplied.  Decided on the host: device code
    // never branches on a pointer's null-ness.
    int has_draft;         // draft logits
    int want_pq;           // diagnostics p_x and q_x
    int want_resid;        // diagnostic resid_mass
    int want_final;        // diagnostic final_row
    // workspace
    uint32_t* err;
    int* next_unit;        // claim counter of the persistent sweep
    // split launches (sv_options.temperature_host): the last split_clusters
    // clusters walk greedy sequences in two halves each; the claim order holds
    // the split_ns sampling sequences first, then the greedy ones, and
    // next_unit_g hands out the greedy queue's tickets after its first wave
    int split_clusters, split_ns;
    int* next_unit_g;
    const int32_t* K;
    const int32_t* order;  // sequences in claim order (longest K first)
    // device copies of K and order in the workspace, filled by the kernel's
    // CTAs at start when the header is in mapped host memory (copy_hdr); a
    // lookup reads them once `ready` counts every CTA, else the header
    int copy_hdr;
    int* ready;
    int32_t* K_dev;
    int32_t* order_dev;
    // ticket c's sequence and its K, c < min(clusters, kFirstUnits): the first
    // wave starts without a claim or a header read
    int32_t first_b[kFirstUnits];
    int32_t first_K[kFirstUnits];
    // logit layout: padded ([B][Kmax+1][V], [B][Kmax][V]) or packed by K
    // (sequence b's rows start at row cu_t[b] of the target and cu_d[b] of the
    // draft array)
    int packed;
    const int32_t* cu_t;
    const int32_t* cu_d;
    // testing: every wait for a slot fill gives up before its first poll
    int expire_waits;
    // small vocabularies (sv_small_kernel): consecutive sequences a warp takes
    int small_tile;
    // per-call counters and the caller's KV lengths (used only if flagged)
    int want_stats, want_kv;
    unsigned long long* stats;   // sv_stats: sequences, invalid, tested, accepted, committed,
                                 // near_ties, draw_near_ties
    int32_t* kv_len;
    // diagnostics (nullable)
    float* p_x;
    float* q_x;
    float* resid;
    int32_t* final_row;
};

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
    // the element's bits, widened to fp32 by widen() where first used, so
    // that no instruction right after the load waits for it
    __device__ static __forceinline__ uint32_t load_raw(const float* p)
    {
        return __float_as_uint(__ldg(p));
    }
    __device__ static __forceinline__ float widen(uint32_t r) { return __uint_as_float(r); }
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
    __device__ static __forceinline__ uint32_t load_raw(const __nv_bfloat16* p)
    {
        uint32_t r;   // 16-bit load, zero-extended into the 32-bit register
        asm("ld.global.nc.u16 %0, [%1];" : "=r"(r) : "l"(p));
        return r;
    }
    __device__ static __forceinline__ float widen(uint32_t r) { return __uint_as_float(r << 16); }
    __device__ static __forceinline__ void copy(__nv_bfloat16* dst, const __nv_bfloat16* src)
    {
        *reinterpret_cast<unsigned short*>(dst) = __ldg(reinterpret_cast<const unsigned short*>(src));
    }
    __device__ static __forceinline__ void set_neg_inf(__nv_bfloat16* dst)
    {
        *reinterpret_cast<unsigned short*>(dst) = 0xFF80u;
    }
};

// c = log2(e) / T, the factor that turns (l - m) into an exp2 argument; one
// correctly rounded fp32 division shared by the sweep and the finaliser.
__device__ __forceinline__ float log2e_over(float T)
{
    return __fdiv_rn(1.44269504088896341f, T);
}

// The unnormalised softmax weight exp2((l - m) c) relative to a reference
// logit m, as exp2(fma(l, c, -r)) with r = m c rounded once: one fused
// multiply-add per element, and every weight of a row carries the same
// rounding of r, which cancels in the ratios p = e / S.  The packed loops
// compute exactly this per element.
__device__ __forceinline__ float ref_of(float m, float c) { return __fmul_rn(m, c); }

__device__ __forceinline__ float weight_r(float l, float r, float c)
{
    return ex2_approx(__fmaf_rn(l, c, -r));
}

__device__ __forceinline__ float weight(float l, float m, float c)
{
    return weight_r(l, ref_of(m, c), c);
}

__device__ __forceinline__ float warp_max_nan(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v = max_nan(v, __shfl_xor_sync(kFull, v, o));
    return v;
}

// Error-free sum: s = fl(a + b) and a + b = s + e exactly (Knuth's TwoSum).
// Symmetric in (a, b), so butterfly partners compute identical pairs.
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e)
{
    s = a + b;
    const float bb = s - a;
    e = (a - (s - bb)) + (b - bb);
}

// Compensated butterfly sum over the warp; every lane ends with the same value.
__device__ __forceinline__ float warp_sum_comp(float v)
{
    float s = v, c = 0.0f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float so = __shfl_xor_sync(kFull, s, o);
        const float co = __shfl_xor_sync(kFull, c, o);
        float t, e;
        two_sum(s, so, t, e);
        s = t;
        c = (c + co) + e;
    }
    return s + c;
}

// Two independent compensated butterfly sums, interleaved so that their
// shuffle latencies overlap; each result equals warp_sum_comp of its input.
__device__ __forceinline__ void warp_sum_comp2(float& va, float& vb)
{
    float sa = va, ca = 0.0f, sb = vb, cb = 0.0f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float soa = __shfl_xor_sync(kFull, sa, o);
        const float sob = __shfl_xor_sync(kFull, sb, o);
        const float coa = __shfl_xor_sync(kFull, ca, o);
        const float cob = __shfl_xor_sync(kFull, cb, o);
        float ta, ea, tb, eb;
        two_sum(sa, soa, ta, ea);
        two_sum(sb, sob, tb, eb);
        sa = ta;
        sb = tb;
        ca = (ca + coa) + ea;
        cb = (cb + cob) + eb;
    }
    va = sa + ca;
    vb = sb + cb;
}

// Two NaN-propagating warp maxima, interleaved.
__device__ __forceinline__ void warp_max_nan2(float& va, float& vb)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float oa = __shfl_xor_sync(kFull, va, o);
        const float ob = __shfl_xor_sync(kFull, vb, o);
        va = max_nan(va, oa);
        vb = max_nan(vb, ob);
    }
}

// Compensated (Neumaier) fp32 running sum.
struct CompSum {
    float s = 0.0f, c = 0.0f;
    __device__ __forceinline__ void add(float v)
    {
        const float t = s + v;
        c += fabsf(s) >= fabsf(v) ? (s - t) + v : (v - t) + s;
        s = t;
    }
    __device__ __forceinline__ float value() const { return s + c; }
};

// Compensated inclusive prefix sum across the warp (lane order): lane l gets
// s + c ~ v_0 + ... + v_l, with the rounding error of the additions kept in c.
__device__ __forceinline__ void warp_incl_scan_comp(float v, int lane, float& s, float& c)
{
    s = v;
    c = 0.0f;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float so = __shfl_up_sync(kFull, s, o);
        const float co = __shfl_up_sync(kFull, c, o);
        if (lane >= o) {
            float t, e;
            two_sum(so, s, t, e);
            s = t;
            c = (co + c) + e;
        }
    }
}

__device__ __forceinline__ bool temperature_usable(float T)
{
    return T == 0.0f || (isfinite(T) && T >= FLT_MIN);
}


}  // namespace sv
