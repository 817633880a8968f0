// Device and host pieces shared by the library's CUDA translation units:
// element-type access (binary16, bfloat16, binary32 in 16-byte words),
// programmatic dependent launch, the fixed-order block reductions and the
// deterministic end of a norm pass, the step-decision kernel, and the host
// helpers that size grids, launch kernels and check arguments.
//
// Everything is in an unnamed namespace: each translation unit that
// includes this header gets its own copy, so no symbol crosses units.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <unordered_map>

#include "zero_pml_internal.h"

namespace zpml {
namespace {

constexpr int kWarps = kThreads / 32;

// ------------------------------------------------------------- element types

template <int DT>
struct Elem;

// binary16: 8 elements in one 16-byte word group
template <>
struct Elem<ZERO_F16> {
    static constexpr int kWords = 1;
    static constexpr int kBytes = 2;
    __device__ static __forceinline__ void to_float(const uint4 *w, float *f)
    {
        const __half2 *h = reinterpret_cast<const __half2 *>(w);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float2 x = __half22float2(h[k]);
            f[2 * k] = x.x;
            f[2 * k + 1] = x.y;
        }
    }
    // A binary16 is inf or NaN iff its exponent field is all ones: adding
    // 0x0400 to the masked field carries into bit 15 exactly then.
    __device__ static __forceinline__ uint32_t nonfinite(const uint4 *w)
    {
        const uint32_t a = ((w->x & 0x7C007C00u) + 0x04000400u) | ((w->y & 0x7C007C00u) + 0x04000400u) |
                           ((w->z & 0x7C007C00u) + 0x04000400u) | ((w->w & 0x7C007C00u) + 0x04000400u);
        return a & 0x80008000u;
    }
    // magnitude bits of the 8 elements ORed: zero iff every element is +-0
    __device__ static __forceinline__ uint32_t nonzero(const uint4 *w)
    {
        return (w->x | w->y | w->z | w->w) & 0x7FFF7FFFu;
    }
    __device__ static __forceinline__ float scalar(const void *p, int64_t i)
    {
        return __half2float(static_cast<const __half *>(p)[i]);
    }
    __device__ static __forceinline__ uint32_t scalar_nonfinite(const void *p, int64_t i)
    {
        return (static_cast<const uint16_t *>(p)[i] & 0x7C00u) == 0x7C00u;
    }
};

// bfloat16: exponent field 0x7F80
template <>
struct Elem<ZERO_BF16> {
    static constexpr int kWords = 1;
    static constexpr int kBytes = 2;
    __device__ static __forceinline__ void to_float(const uint4 *w, float *f)
    {
        const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(w);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float2 x = __bfloat1622float2(h[k]);
            f[2 * k] = x.x;
            f[2 * k + 1] = x.y;
        }
    }
    __device__ static __forceinline__ uint32_t nonfinite(const uint4 *w)
    {
        const uint32_t a = ((w->x & 0x7F807F80u) + 0x00800080u) | ((w->y & 0x7F807F80u) + 0x00800080u) |
                           ((w->z & 0x7F807F80u) + 0x00800080u) | ((w->w & 0x7F807F80u) + 0x00800080u);
        return a & 0x80008000u;
    }
    __device__ static __forceinline__ uint32_t nonzero(const uint4 *w)
    {
        return (w->x | w->y | w->z | w->w) & 0x7FFF7FFFu;
    }
    __device__ static __forceinline__ float scalar(const void *p, int64_t i)
    {
        return __bfloat162float(static_cast<const __nv_bfloat16 *>(p)[i]);
    }
    __device__ static __forceinline__ uint32_t scalar_nonfinite(const void *p, int64_t i)
    {
        return (static_cast<const uint16_t *>(p)[i] & 0x7F80u) == 0x7F80u;
    }
};

// binary32: 8 elements in two 16-byte words
template <>
struct Elem<ZERO_F32> {
    static constexpr int kWords = 2;
    static constexpr int kBytes = 4;
    __device__ static __forceinline__ void to_float(const uint4 *w, float *f)
    {
        f[0] = __uint_as_float(w[0].x);
        f[1] = __uint_as_float(w[0].y);
        f[2] = __uint_as_float(w[0].z);
        f[3] = __uint_as_float(w[0].w);
        f[4] = __uint_as_float(w[1].x);
        f[5] = __uint_as_float(w[1].y);
        f[6] = __uint_as_float(w[1].z);
        f[7] = __uint_as_float(w[1].w);
    }
    __device__ static __forceinline__ uint32_t nonfinite(const uint4 *w)
    {
        uint32_t a = 0;
#pragma unroll
        for (int q = 0; q < 2; ++q)
            a |= ((w[q].x & 0x7F800000u) + 0x00800000u) | ((w[q].y & 0x7F800000u) + 0x00800000u) |
                 ((w[q].z & 0x7F800000u) + 0x00800000u) | ((w[q].w & 0x7F800000u) + 0x00800000u);
        return a & 0x80000000u;
    }
    __device__ static __forceinline__ uint32_t nonzero(const uint4 *w)
    {
        return (w[0].x | w[0].y | w[0].z | w[0].w | w[1].x | w[1].y | w[1].z | w[1].w) & 0x7FFFFFFFu;
    }
    __device__ static __forceinline__ float scalar(const void *p, int64_t i)
    {
        return static_cast<const float *>(p)[i];
    }
    __device__ static __forceinline__ uint32_t scalar_nonfinite(const void *p, int64_t i)
    {
        return (__float_as_uint(static_cast<const float *>(p)[i]) & 0x7F800000u) == 0x7F800000u;
    }
};

// Low-precision parameter copy: binary32 -> 16-bit, round to nearest even.
template <int PT>
struct LowP;

template <>
struct LowP<ZERO_F16> {
    __device__ static __forceinline__ uint4 pack(const float *f)
    {
        uint4 r;
        __half2 h0 = __floats2half2_rn(f[0], f[1]), h1 = __floats2half2_rn(f[2], f[3]);
        __half2 h2 = __floats2half2_rn(f[4], f[5]), h3 = __floats2half2_rn(f[6], f[7]);
        r.x = *reinterpret_cast<uint32_t *>(&h0);
        r.y = *reinterpret_cast<uint32_t *>(&h1);
        r.z = *reinterpret_cast<uint32_t *>(&h2);
        r.w = *reinterpret_cast<uint32_t *>(&h3);
        return r;
    }
    __device__ static __forceinline__ void store(void *p, int64_t i, float x)
    {
        static_cast<__half *>(p)[i] = __float2half_rn(x);
    }
};

template <>
struct LowP<ZERO_BF16> {
    __device__ static __forceinline__ uint4 pack(const float *f)
    {
        uint4 r;
        __nv_bfloat162 h0 = __floats2bfloat162_rn(f[0], f[1]), h1 = __floats2bfloat162_rn(f[2], f[3]);
        __nv_bfloat162 h2 = __floats2bfloat162_rn(f[4], f[5]), h3 = __floats2bfloat162_rn(f[6], f[7]);
        r.x = *reinterpret_cast<uint32_t *>(&h0);
        r.y = *reinterpret_cast<uint32_t *>(&h1);
        r.z = *reinterpret_cast<uint32_t *>(&h2);
        r.w = *reinterpret_cast<uint32_t *>(&h3);
        return r;
    }
    __device__ static __forceinline__ void store(void *p, int64_t i, float x)
    {
        static_cast<__nv_bfloat16 *>(p)[i] = __float2bfloat16_rn(x);
    }
};

// ------------------------------------------------------------- launch order

// Programmatic dependent launch.  A kernel launched with the programmatic
// stream-serialisation attribute may be scheduled while the kernel before it
// in the stream is still running; pdl_wait() blocks until that kernel (and
// so all earlier work in the stream) has completed and its writes are
// visible, and must come before the first access to memory produced
// earlier.  For a kernel launched without the attribute it returns at once.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Allows the next kernel in the stream to be scheduled now (it still waits
// in pdl_wait() for this one to finish).  Used only by kernels whose
// successor needs few SM slots while it waits.
__device__ __forceinline__ void pdl_launch_next() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ------------------------------------------------------------- bulk copies

// Bulk asynchronous copies from global into shared memory (cp.async.bulk,
// the untiled TMA copy) that complete on an mbarrier: the issuing thread
// arms the barrier with the byte count, the copy engine counts the bytes
// down, and the barrier's phase flips when all have landed.  Both addresses
// are 16-byte aligned and the size a multiple of 16.

__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return (uint32_t)__cvta_generic_to_shared(p);
}

// Nanoseconds of the GPU's global timer (for wait limits).
__device__ __forceinline__ uint64_t global_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// One-thread set-up of `count` barriers expecting one arrival each, made
// visible to the copy engine (async proxy) before the first copy.
__device__ __forceinline__ void mbar_init(uint64_t *bars, int count)
{
    for (int s = 0; s < count; ++s)
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(bars + s)) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Waits for the phase of parity `parity` of a barrier to complete, until the
// global timer passes `deadline_ns`; false if it gave up.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, uint64_t deadline_ns)
{
    for (uint32_t it = 0;; ++it) {
        uint32_t done;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(done)
            : "r"(smem_addr(bar)), "r"(parity)
            : "memory");
        if (done)
            return true;
        if ((it & 63u) == 63u && global_ns() > deadline_ns)
            return false;
    }
}

// L2 eviction priorities for a copy's lines: evict-last keeps them for a
// later kernel, evict-first lets a stream pass through.
__device__ __forceinline__ uint64_t l2_policy(bool keep)
{
    uint64_t pol;
    if (keep)
        asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    else
        asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// Arms `bar` for `bytes` and starts the copy of [src, src + bytes) into
// shared memory at dst (one thread).  Before reusing a buffer that threads
// have read, the issuing thread orders those reads before the copy's writes
// with fence.proxy.async (after a block barrier).
__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes, uint64_t *bar, uint64_t policy)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::
            "r"(smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// ------------------------------------------------------------- reductions

__device__ __forceinline__ double warp_sum(double x)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// binary32 sum of 8 lanes in a fixed tree
__device__ __forceinline__ float tree8(const float *a)
{
    return __fadd_rn(__fadd_rn(__fadd_rn(a[0], a[1]), __fadd_rn(a[2], a[3])),
                     __fadd_rn(__fadd_rn(a[4], a[5]), __fadd_rn(a[6], a[7])));
}

// ------------------------------------------------------------- squares in range
//
// The norm passes square in binary32 and add each 8-element vector's squares
// in a fixed binary32 tree before they reach the binary64 total.  Binary16
// data always fits: |x| <= 65504 and every nonzero binary16 is at least
// 2^-24, so every square is a normal binary32 between 2^-48 and 2^32.
// Bfloat16 and binary32 data span binary32's whole range: a square
// overflows to inf once |x| passes 2^64, and falls below the normal range
// (losing digits, or vanishing) once |x| drops under 2^-63.  For those types
// each vector's binary32 sum s is checked before use: it is kept if
// s < 2^124 (then four such sums still add without overflow) and either
// s >= 2^-90 (a square under 2^-126 then changes s by less than 2^-33 of
// itself) or all eight values are zero.  Otherwise -- a value above about
// 2^62, an inf or NaN, or a vector of tiny values -- the vector's squares are
// summed again in binary64, which neither overflows nor underflows for any
// binary32 value.  Typical data never leaves the fast path.

// Magnitude bits of 8 binary32 values ORed: zero iff every value is +-0.
__device__ __forceinline__ uint32_t nonzero8(const float *f)
{
    uint32_t b = 0;
#pragma unroll
    for (int e = 0; e < 8; ++e)
        b |= __float_as_uint(f[e]);
    return b & 0x7FFFFFFFu;
}

// Whether the binary32 sum s of a vector's squares may be used (see above).
__device__ __forceinline__ bool squares_in_range(float s, uint32_t nonzero)
{
    return s < 0x1p124f && (s >= 0x1p-90f || nonzero == 0u);
}

// The vector's squares summed in binary64.
__device__ __forceinline__ double squares_wide(const float *f)
{
    double t = 0.0;
#pragma unroll
    for (int e = 0; e < 8; ++e)
        t = __fma_rn((double)f[e], (double)f[e], t);
    return t;
}

// The squares of one vector (8 values f, whose magnitude bits OR to
// `nonzero`) added to a binary32 partial `part`, or -- out of range -- to
// the binary64 total `tot`.
__device__ __forceinline__ void add_squares_checked(const float *f, uint32_t nonzero, float &part, double &tot)
{
    float sq[8];
#pragma unroll
    for (int e = 0; e < 8; ++e)
        sq[e] = __fmul_rn(f[e], f[e]);
    const float s = tree8(sq);
    if (squares_in_range(s, nonzero))
        part = __fadd_rn(part, s);
    else
        tot += squares_wide(f);
}

// Block sum (fixed order) of a per-thread binary64 value and OR of a flag.
// Result valid in thread 0.
__device__ __forceinline__ void block_reduce(double &tot, uint32_t &bad)
{
    __shared__ double s_tot[kWarps];
    __shared__ uint32_t s_bad[kWarps];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    tot = warp_sum(tot);
    const uint32_t b = __any_sync(0xffffffffu, bad != 0);
    if (lane == 0) {
        s_tot[warp] = tot;
        s_bad[warp] = b;
    }
    __syncthreads();
    if (warp == 0) {
        double t = lane < kWarps ? s_tot[lane] : 0.0;
        const uint32_t bb = __any_sync(0xffffffffu, lane < kWarps && s_bad[lane] != 0);
        tot = warp_sum(t);
        bad = bb;
    }
    __syncthreads();
}

// Shared-memory copies of the state and of the bias-correction cache, the
// inputs of the decision: loaded by the block together with what it waits
// for anyway (the partials of the norm), so that the decision issues no
// dependent global load of its own.
struct DecideShared {
    zero_state_t s;
    PowCache c;
};

// Block code: the state and (if `cache` is not NULL) the cache into `sh`,
// 8 bytes per thread; visible after the caller's next barrier.
__device__ __forceinline__ void decide_load(const zero_state_t *st, const PowCache *cache, DecideShared *sh)
{
    constexpr int kS = sizeof(zero_state_t) / 8, kC = sizeof(PowCache) / 8;
    static_assert(sizeof(zero_state_t) % 8 == 0 && sizeof(PowCache) % 8 == 0, "8-byte words");
    const int k = threadIdx.x;
    if (k < kS)
        reinterpret_cast<uint64_t *>(&sh->s)[k] = reinterpret_cast<const uint64_t *>(st)[k];
    else if (cache && k < kS + kC)
        reinterpret_cast<uint64_t *>(&sh->c)[k - kS] = reinterpret_cast<const uint64_t *>(cache)[k - kS];
}

// 1 / S for the loss scale S.  S is a power of two (the initial scale is
// checked, and it is only ever halved or doubled): its reciprocal is then
// exact, the exponent negated with a zero fraction, which spares the slow
// binary64 division; any other value takes the division.
__device__ __forceinline__ double inverse_scale(double x)
{
    const long long b = __double_as_longlong(x);
    if ((b & 0x000FFFFFFFFFFFFFLL) == 0 && b >= 0x3FF0000000000000LL && b <= 0x7FD0000000000000LL)
        return __longlong_as_double(0x7FE0000000000000LL - b);
    return 1.0 / x;
}

// End of the norm pass in every block: publish this block's partial; the
// block that takes the last ticket sums all partials in block order and
// writes (or adds) the unscaled totals into the state.  No block waits on
// another: the last block to arrive does the final sum.  Returns true in
// every thread of that last block.
__device__ bool norm_finish(double tot, uint32_t bad, double2 *partials, WsHeader *hdr,
                            zero_state_t *st, int accumulate, DecideShared *sh, const PowCache *cache = nullptr)
{
    __shared__ bool s_last;
    block_reduce(tot, bad);
    if (threadIdx.x == 0) {
        partials[blockIdx.x] = make_double2(tot, bad ? 1.0 : 0.0);
        __threadfence();
        const unsigned int ticket = atomicAdd(&hdr->ticket, 1u);
        s_last = (ticket == gridDim.x - 1);
    }
    __syncthreads();
    if (!s_last)
        return false;
    __threadfence();
    // the state (and the cache, for a decision taken here) beside the partials
    decide_load(st, cache, sh);
    double t = 0.0;
    uint32_t b = 0;
    for (int j = threadIdx.x; j < (int)gridDim.x; j += kThreads) {
        const double2 q = __ldcg(partials + j);
        t += q.x;
        b |= (q.y != 0.0);
    }
    block_reduce(t, b);
    if (threadIdx.x == 0) {
        // the partials hold sums of squares of the stored (scaled) gradient;
        // the loss scale is a power of two, so this rescaling is exact
        const double inv = inverse_scale(sh->s.loss_scale);
        const double sum = t * inv * inv;
        sh->s.sumsq = accumulate ? sh->s.sumsq + sum : sum;
        sh->s.found_inf = (accumulate ? sh->s.found_inf : 0.0) + (b ? 1.0 : 0.0);
        st->sumsq = sh->s.sumsq;
        st->found_inf = sh->s.found_inf;
        hdr->ticket = 0u;
    }
    return true;
}

// The end of a one-shot reduction (one partial per block, any number of
// blocks up to kGroupBlocks * kMaxGroups), deterministic and without any
// block waiting on another: each block publishes its partial; the last block
// of its group of kGroupBlocks sums the group's partials in block order; the
// last group to finish sums the group partials in group order.  Returns true
// in thread 0 of that final block, with the grand totals in tot and bad.
__device__ bool group_finish(double &tot, uint32_t &bad, double2 *block_partials, GroupArea *ga, WsHeader *hdr)
{
    __shared__ bool s_flag;
    block_reduce(tot, bad);
    const unsigned g = blockIdx.x / kGroupBlocks;
    const unsigned g0 = g * kGroupBlocks;
    const unsigned gsize = gridDim.x - g0 < (unsigned)kGroupBlocks ? gridDim.x - g0 : (unsigned)kGroupBlocks;
    const unsigned ngroups = (gridDim.x + kGroupBlocks - 1) / kGroupBlocks;
    double2 *gpart = reinterpret_cast<double2 *>(ga->partials);
    if (threadIdx.x == 0) {
        block_partials[blockIdx.x] = make_double2(tot, bad ? 1.0 : 0.0);
        __threadfence();
        s_flag = atomicAdd(&ga->tickets[g], 1u) == gsize - 1;
    }
    __syncthreads();
    if (!s_flag)
        return false;
    __threadfence();
    double t = 0.0;
    uint32_t b = 0;
    for (unsigned j = threadIdx.x; j < gsize; j += kThreads) {
        const double2 q = __ldcg(block_partials + g0 + j);
        t += q.x;
        b |= (q.y != 0.0);
    }
    block_reduce(t, b);
    if (threadIdx.x == 0) {
        ga->tickets[g] = 0u;
        gpart[g] = make_double2(t, b ? 1.0 : 0.0);
        __threadfence();
        s_flag = atomicAdd(&hdr->ticket, 1u) == ngroups - 1;
    }
    __syncthreads();
    if (!s_flag)
        return false;
    __threadfence();
    t = 0.0;
    b = 0;
    for (unsigned j = threadIdx.x; j < ngroups; j += kThreads) {
        const double2 q = __ldcg(gpart + j);
        t += q.x;
        b |= (q.y != 0.0);
    }
    block_reduce(t, b);
    if (threadIdx.x != 0)
        return false;
    hdr->ticket = 0u;
    tot = t;
    bad = b;
    return true;
}

// The squared norm and overflow of a reduction pass written into the state:
// the partials hold sums of squares of the stored (scaled) gradient; the loss
// scale is a power of two, so the rescaling is exact.
__device__ __forceinline__ void write_norm(zero_state_t *st, double tot, uint32_t bad, int accumulate)
{
    const double inv = 1.0 / st->loss_scale;
    const double sum = tot * inv * inv;
    st->sumsq = accumulate ? st->sumsq + sum : sum;
    st->found_inf = (accumulate ? st->found_inf : 0.0) + (bad ? 1.0 : 0.0);
}

// ------------------------------------------------------------- decision

struct DecideArgs {
    double lr, beta1, beta2, max_norm, min_scale;
    int64_t scale_window;
    // step scalars that do not depend on the device state, computed on the
    // host the same way (binary64, rounded once to binary32)
    float b1, omb1, b2, omb2, eps, lrwd;
    // 1-bit Adam's compression stage: the variance and its bias correction
    // are frozen at the last warm-up step; isb2 is then that step's value
    int32_t frozen;
    float isb2_frozen;
};

// Hyper-parameters in range: lr, eps, weight decay >= 0, betas in [0, 1),
// a scale floor >= 1, a growth window >= 1, max_norm not NaN.
// The floor of the loss scale is a power of two like the scale itself, so
// that halving down to it keeps the scale a power of two.
inline bool hparams_ok(const zero_hparams_t *hp)
{
    int e = 0;
    return hp->lr >= 0.0 && hp->beta1 >= 0.0 && hp->beta1 < 1.0 && hp->beta2 >= 0.0 && hp->beta2 < 1.0 &&
           hp->eps >= 0.0 && hp->weight_decay >= 0.0 && hp->min_scale >= 1.0 && std::isfinite(hp->min_scale) &&
           std::frexp(hp->min_scale, &e) == 0.5 && hp->scale_window >= 1 && hp->max_norm == hp->max_norm;
}

// The decision's arguments from the host hyper-parameters; freeze_step > 0
// freezes the variance correction at 1/sqrt(1 - beta2^freeze_step).
inline DecideArgs decide_args(const zero_hparams_t *hp, int64_t freeze_step = 0)
{
    DecideArgs a;
    a.lr = hp->lr;
    a.beta1 = hp->beta1;
    a.beta2 = hp->beta2;
    a.max_norm = hp->max_norm;
    a.min_scale = hp->min_scale;
    a.scale_window = hp->scale_window;
    a.b1 = (float)hp->beta1;
    a.omb1 = (float)(1.0 - hp->beta1);
    a.b2 = (float)hp->beta2;
    a.omb2 = (float)(1.0 - hp->beta2);
    a.eps = (float)hp->eps;
    a.lrwd = (float)(hp->lr * hp->weight_decay);
    a.frozen = freeze_step > 0;
    a.isb2_frozen = a.frozen ? (float)(1.0 / std::sqrt(1.0 - std::pow(hp->beta2, (double)freeze_step))) : 0.0f;
    return a;
}

// Thread 0's part of the decision: the skip, the loss scale and counters,
// and the step scalars from the three chains' results.
__device__ __forceinline__ void decide_write(zero_state_t *st, StepScalars *out, const DecideArgs &a, zero_state_t s,
                                             const float *s_val, double norm)
{
    StepScalars o;
    // S is a power of two: below 2^127 its binary32 reciprocal is exact and
    // equals the binary64 reciprocal rounded to binary32
    o.inv_scale = s.loss_scale <= 0x1p126 ? __frcp_rn((float)s.loss_scale) : (float)(1.0 / s.loss_scale);
    o.clip = 1.0f;
    o.b1 = o.omb1 = o.b2 = o.omb2 = o.eps = o.step_size = o.isb2 = o.lrwd = 0.0f;
    o.pad = 0;
    if (s.found_inf != 0.0) {
        o.skip = 1;
        const double half = s.loss_scale * 0.5;
        s.loss_scale = half < a.min_scale ? a.min_scale : half;
        s.good_steps = 0;
        s.skipped += 1;
    } else {
        o.skip = 0;
        s.step += 1;
        s.good_steps += 1;
        if (s.good_steps >= a.scale_window) {
            s.loss_scale *= 2.0;
            s.good_steps = 0;
        }
        o.clip = s_val[2];
        o.b1 = a.b1;
        o.omb1 = a.omb1;
        o.b2 = a.b2;
        o.omb2 = a.omb2;
        o.eps = a.eps;
        o.step_size = s_val[0];
        o.isb2 = s_val[1];
        o.lrwd = a.lrwd;
    }
    o.lr = a.lr;
    o.beta1 = a.beta1;
    o.beta2 = a.beta2;
    o.next_t = s.step + 1;
    s.last_norm = norm;
    s.last_clip = o.clip;
    s.last_skipped = o.skip;
    s.sumsq = 0.0;
    s.found_inf = 0.0;
    *st = s;
    *out = o;
}


// Skip or apply, loss-scale and step bookkeeping, and the step scalars
// (binary64, each rounded once to binary32).  Binary64 is a slow pipe on
// this GPU, so the independent chains run side by side: lanes 0 and 1 of
// warp 0 take 1 - beta1^t with the step size and 1 - beta2^t with its
// inverse square root (from the cache window when its tags match, else one
// converged pow each), warp 1 the norm and the clip coefficient; thread 0
// then writes the results.  Block code: every thread of the block (at
// least 64) calls it (it holds a block barrier).
__device__ __forceinline__ void decide_block(zero_state_t *st, StepScalars *out, const DecideShared &sh,
                                             const DecideArgs &a)
{
    __shared__ float s_val[3];
    __shared__ double s_norm;
    const int tid = threadIdx.x;
    const zero_state_t &s = sh.s;
    const PowCache &c = sh.c;
    const int64_t tn = s.step + 1;  // the step count if this step applies
    if (tid < 2) {
        const bool hit = c.t0 > 0 && tn >= c.t0 && tn < c.t0 + kPowWindow && c.beta1 == a.beta1 &&
                         c.beta2 == a.beta2;
        const int j = hit ? (int)(tn - c.t0) : 0;
        if (tid == 0 && hit && c.lr == a.lr) {
            s_val[0] = c.step_size[j];
        } else if (tid == 1 && (a.frozen || hit)) {
            s_val[1] = a.frozen ? a.isb2_frozen : c.isb2[j];
        } else {
            // the cache's expressions, evaluated here
            const double bc = tid == 0 && hit ? c.bc1[j] : 1.0 - pow(tid ? a.beta2 : a.beta1, (double)tn);
            s_val[tid] = tid ? (float)(1.0 / sqrt(bc)) : (float)(a.lr / bc);
        }
    } else if (tid == 32) {
        const double norm = sqrt(s.sumsq);
        double clip = 1.0;
        if (a.max_norm > 0.0) {
            const double q = a.max_norm / (norm + 1e-6);
            if (q < 1.0)
                clip = q;
        }
        s_norm = norm;
        s_val[2] = (float)clip;
    }
    __syncthreads();
    if (tid == 0)
        decide_write(st, out, a, s, s_val, s_norm);
}

// The step's scalars, read after the decision wrote them.  One volatile
// 16-byte load per word: a kernel launched with programmatic dependent
// launch must not read them before its griddepcontrol.wait (which makes the
// previous kernel's writes visible), and the compiler may move a plain load
// of memory it takes for read-only (a const __restrict__ pointer) above
// that wait; an asm volatile load stays in program order with it.  The load
// may be served by L1: every warp of the grid reads these 80 bytes, and
// sent to L2 each time (ld.global.cg) they made one L2 slice the step's
// bottleneck (a 1.56G-element step took 10.1 ms instead of 6.56).
__device__ __forceinline__ StepScalars load_scalars(const StepScalars *p)
{
    static_assert(sizeof(StepScalars) % 16 == 0, "StepScalars is read in 16-byte words");
    StepScalars s;
    uint4 *d = reinterpret_cast<uint4 *>(&s);
    const uint4 *q = reinterpret_cast<const uint4 *>(p);
#pragma unroll
    for (int k = 0; k < (int)(sizeof(StepScalars) / 16); ++k)
        asm volatile("ld.global.v4.u32 {%0,%1,%2,%3}, [%4];"
                     : "=r"(d[k].x), "=r"(d[k].y), "=r"(d[k].z), "=r"(d[k].w)
                     : "l"(q + k)
                     : "memory");
    return s;
}

// The bias-correction window for the next applied step, if the cache does
// not cover it: warp code (all 32 lanes of one warp), lanes 0..15 taking
// 1 - beta1^t and lanes 16..31 1 - beta2^t for t = next_t .. next_t + 15 in
// one converged pow.  The same expressions as the decision's own.  A change
// of the learning rate alone refills nothing: the decision then divides the
// new rate by the cached 1 - beta1^t (a schedule changes it every step).
__device__ __forceinline__ void refill_pow_window(const StepScalars &sc, PowCache *cache)
{
    const int lane = threadIdx.x & 31;
    const int64_t tn = sc.next_t;
    const double lr = sc.lr, beta1 = sc.beta1, beta2 = sc.beta2;
    if (cache->t0 > 0 && tn >= cache->t0 && tn < cache->t0 + kPowWindow && cache->beta1 == beta1 &&
        cache->beta2 == beta2)
        return;
    const int j = lane & (kPowWindow - 1);
    const double bc = 1.0 - pow(lane < kPowWindow ? beta1 : beta2, (double)(tn + j));
    if (lane < kPowWindow) {
        cache->bc1[j] = bc;
        cache->step_size[j] = (float)(lr / bc);
    } else {
        cache->isb2[j] = (float)(1.0 / sqrt(bc));
    }
    if (lane == 0) {
        cache->t0 = tn;
        cache->beta1 = beta1;
        cache->beta2 = beta2;
        cache->lr = lr;
    }
}

// The decision as a kernel of one block of 64 threads.  `refill`: then
// also the bias-correction window for the next step (warp 0, after the
// decision), for callers whose streaming kernels do not refill it.
__global__ void k_decide(zero_state_t *st, StepScalars *out, PowCache *cache, DecideArgs a, int refill)
{
    pdl_launch_next();
    pdl_wait();
    if (blockIdx.x != 0)
        return;
    __shared__ DecideShared sh;
    decide_load(st, cache, &sh);
    __syncthreads();
    decide_block(st, out, sh, a);
    if (!refill)
        return;
    __syncthreads();
    if (threadIdx.x < 32) {
        const StepScalars o = load_scalars(out);
        if (!o.skip)
            refill_pow_window(o, cache);
    }
}
// ------------------------------------------------------------- host helpers

int sm_count()
{
    static std::mutex mu;
    static std::unordered_map<int, int> cache;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return 0;
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(dev);
    if (it != cache.end())
        return it->second;
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 0;
    cache[dev] = v;
    return v;
}

// Resident blocks per SM of a kernel at kThreads threads (cached per device
// and kernel).
int blocks_per_sm(const void *kernel)
{
    static std::mutex mu;
    static std::unordered_map<uint64_t, int> cache;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return 1;
    const uint64_t key = reinterpret_cast<uint64_t>(kernel) ^ ((uint64_t)dev << 56);
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(key);
    if (it != cache.end())
        return it->second;
    int b = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, kernel, kThreads, 0) != cudaSuccess || b < 1)
        b = 1;
    cache[key] = b;
    return b;
}

// A whole number of waves over the SMs (at most per_sm_cap blocks per SM), or
// fewer blocks if there is less work.
int grid_for(const void *kernel, int64_t work_items, int cap, int per_sm_cap = 1 << 30)
{
    const int bps = blocks_per_sm(kernel);
    const int64_t full = (int64_t)sm_count() * (bps < per_sm_cap ? bps : per_sm_cap);
    int64_t g = work_items < full ? work_items : full;
    if (g > cap)
        g = cap;
    return g < 1 ? 1 : (int)g;
}

// Launches a kernel; with `pdl` set, with programmatic stream
// serialisation, so that it can be scheduled while the previous kernel in
// the stream finishes (the kernel itself waits in pdl_wait() before touching
// memory).  The wait covers the previous KERNEL only: `pdl` is set only where
// the previous operation in the stream is this library's own kernel of the
// same call -- never after a copy, a memset or the caller's work.
template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*kernel)(KArgs...), int grid, int block, cudaStream_t stream, bool pdl, Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3((unsigned)block);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

int check_launch(const char *what)
{
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        set_cuda_error(what, (int)e, cudaGetErrorString(e));
        return ZERO_ECUDA;
    }
    return ZERO_OK;
}

// Copies a host-built table into the workspace without stalling the host.
// A copy from pageable memory makes the host wait until the stream has
// drained, which leaves the GPU idle between consecutive calls; the table is
// therefore staged through one of two pinned host buffers per device,
// allocated on first use and grown as needed, each reused only once the
// copy out of it two uploads ago has completed (an event, long past by
// then).  If pinned memory cannot be had, the copy goes from pageable memory.
cudaError_t stage_copy(void *dst, const void *src, size_t bytes, cudaStream_t stream)
{
    struct Ring {
        void *buf[2] = {nullptr, nullptr};
        size_t cap[2] = {0, 0};
        cudaEvent_t ev[2] = {nullptr, nullptr};
        int next = 0;
    };
    static std::mutex mu;
    static std::unordered_map<int, Ring> rings;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    std::lock_guard<std::mutex> lock(mu);
    Ring &r = rings[dev];
    const int k = r.next;
    r.next ^= 1;
    if (r.ev[k] && (e = cudaEventSynchronize(r.ev[k])) != cudaSuccess)
        return e;
    if (r.cap[k] < bytes) {
        if (r.buf[k])
            cudaFreeHost(r.buf[k]);
        r.buf[k] = nullptr;
        r.cap[k] = 0;
        const size_t want = bytes + bytes / 2;
        if (cudaHostAlloc(&r.buf[k], want, cudaHostAllocDefault) == cudaSuccess) {
            r.cap[k] = want;
        } else {
            cudaGetLastError();
            r.buf[k] = nullptr;
            return cudaMemcpyAsync(dst, src, bytes, cudaMemcpyHostToDevice, stream);
        }
    }
    std::memcpy(r.buf[k], src, bytes);
    if ((e = cudaMemcpyAsync(dst, r.buf[k], bytes, cudaMemcpyHostToDevice, stream)) != cudaSuccess)
        return e;
    if (!r.ev[k] && (e = cudaEventCreateWithFlags(&r.ev[k], cudaEventDisableTiming)) != cudaSuccess)
        return e;
    return cudaEventRecord(r.ev[k], stream);
}

// The table copy of a call, or ZERO_ECAPTURE with nothing enqueued while
// `stream` is being captured into a graph: a captured copy would read the
// staging buffer when the graph is replayed, after later calls have reused
// it.  Returns ZERO_OK, ZERO_ECAPTURE or ZERO_ECUDA (the message under `what`).
int stage_upload(void *dst, const void *src, size_t bytes, cudaStream_t stream, const char *what)
{
    if (bytes == 0)
        return ZERO_OK;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(stream, &cs);
    if (e == cudaSuccess && cs != cudaStreamCaptureStatusNone)
        return ZERO_ECAPTURE;
    if (e == cudaSuccess)
        e = stage_copy(dst, src, bytes, stream);
    if (e != cudaSuccess) {
        cudaGetLastError();
        set_cuda_error(what, (int)e, cudaGetErrorString(e));
        return ZERO_ECUDA;
    }
    return ZERO_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool grad_dtype_ok(int32_t d) { return d == ZERO_F16 || d == ZERO_BF16 || d == ZERO_F32; }
bool lp_dtype_ok(int32_t d) { return d == ZERO_F16 || d == ZERO_BF16; }

// True when the pointer is device memory the kernels may stream (device or
// managed allocations).  Host memory is refused even where the GPU could
// reach it: the kernels assume HBM.
bool device_ptr(const void *p)
{
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged;
}

// True for plain device memory (cudaMalloc), the only memory the kernels
// read with bulk asynchronous copies: managed or host memory takes the
// paths that use ordinary loads.
bool plain_device_ptr(const void *p)
{
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return a.type == cudaMemoryTypeDevice;
}

// True for memory the kernels may reach that lives in host memory: pinned
// (cudaHostAlloc / cudaHostRegister) allocations, mapped into the device
// address space.  On GB300 the kernels reach it over NVLink-C2C.
bool pinned_host_ptr(const void *p)
{
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return a.type == cudaMemoryTypeHost && a.devicePointer == p;
}

// Lists up to this many arrays have every array's pointer checked to be
// memory the kernels may reach.
constexpr int64_t kCheckEveryPointer = 64;

// Checks one list; on success *total holds its element count.  The device
// pointers of a list of up to kCheckEveryPointer arrays are each checked to
// be device memory (or, with allow_host, pinned host memory); longer lists
// are checked on their first and last arrays only, to keep the per-call host
// cost independent of the list length (a few hundred nanoseconds per check).
int check_list(const zero_tlist_t *l, int64_t *total, bool allow_host = false)
{
    if (!l || l->n < 0 || (l->n > 0 && (!l->ptrs || !l->numel)))
        return ZERO_EINVAL;
    int64_t t = 0;
    for (int64_t i = 0; i < l->n; ++i) {
        if (l->numel[i] < 0)
            return ZERO_EINVAL;
        if (l->numel[i] > 0) {
            if (!l->ptrs[i])
                return ZERO_EINVAL;
            if (!aligned16(l->ptrs[i]))
                return ZERO_EALIGN;
        }
        t += l->numel[i];
    }
    for (int64_t i = 0; i < l->n; ++i) {
        if (l->n > kCheckEveryPointer && i > 0 && i < l->n - 1)
            i = l->n - 1;
        if (l->numel[i] > 0 && !device_ptr(l->ptrs[i]) && !(allow_host && pinned_host_ptr(l->ptrs[i])))
            return ZERO_EINVAL;
    }
    *total = t;
    return ZERO_OK;
}

int check_same_shape(const zero_tlist_t *a, const zero_tlist_t *b)
{
    if (a->n != b->n)
        return ZERO_ESIZE;
    for (int64_t i = 0; i < a->n; ++i)
        if (a->numel[i] != b->numel[i])
            return ZERO_ESIZE;
    return ZERO_OK;
}

int check_ws(void *ws, size_t ws_bytes, int64_t n_tensors, int64_t total)
{
    if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0)
        return ws ? ZERO_EALIGN : ZERO_EWORKSPACE;
    if (ws_bytes < zero_workspace_bytes(n_tensors, total))
        return ZERO_EWORKSPACE;
    if (!device_ptr(ws))
        return ZERO_EINVAL;
    return ZERO_OK;
}

}  // namespace
}  // namespace zpml
