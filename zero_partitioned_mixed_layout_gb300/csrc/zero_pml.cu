// CUDA part of the C ABI (sm_103a): gradient accumulation, pass 1 (unscale,
// overflow, squared norm), the one-thread step decision, and pass 2 (clip,
// AdamW, cast) over one rank's flat shard or over a list of arrays.
//
// Sources: "ZeRO: Memory Optimizations Toward Training Trillion Parameter
// Models - 中文验证版" (ai-papers.xuzou.cn), sections 瓶颈 (bottleneck: the
// mixed-precision Adam state is fp16 param + grad and fp32 master, momentum,
// variance) and 方法适配 (method: each data-parallel rank owns one partition
// of that state and updates only it); DeepSpeed release news
// (lxsoso.com/blog/19320.html): mixed precision and gradient accumulation.
// The update is Adam (Kingma & Ba 2015) with decoupled weight decay
// (Loshchilov & Hutter 2019) and dynamic loss scaling (Micikevicius et al.
// 2018).
//
// Design: every kernel here streams HBM once.  Per element pass 2 reads
// 2 + 12 bytes and writes 12 + 2 bytes (fp16 grad/param): 28 bytes.  Loads
// and stores are 16-byte vectors with streaming cache hints, eight elements
// per thread.  Pass 2 over a flat shard is one-shot (one vector per thread,
// the grid covering the array once); the reductions run on persistent grids
// of 4 blocks per SM.  Consecutive kernels use programmatic dependent launch
// so that each is scheduled while the previous one drains.
// The element arithmetic uses explicit round-to-nearest intrinsics, so no
// multiply-add is ever contracted and the result is the IEEE binary32 value
// of the documented expression, bit for bit.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cuda.h>  // driver types for the context identity (no driver library linked)
#include <cudaTypedefs.h>

#include <cstdint>
#include <mutex>
#include <unordered_map>
#include <vector>

#include "common.cuh"

namespace zpml {
namespace {

// Bytes at the end of a flat gradient that pass 1 asks L2 to keep for pass 2
// (GB300 has 126 MB of L2; pass 2's other streams are evict-first).
constexpr int64_t kL2KeepBytes = 96ll << 20;

// ------------------------------------------------------------- pass 1

// Vectors (of 8 elements) a thread of pass 1 loads at a time.
constexpr int kNormVectors = 4;

// Squares of kNormVectors vectors in 8 binary32 lanes, then one binary64
// add per thread: the binary64 pipe sees one add per 8 * kNormVectors
// elements.  Binary16: every square is a normal binary32.  Bfloat16 and
// binary32: the group's binary32 sum is kept only if it is finite (then no
// square or lane sum overflowed) and either at least 2^-90 (squares lost
// below binary32's normal range then change it by less than 2^-31 of
// itself) or every value is zero; otherwise the group, still in registers,
// is summed again in binary64.
template <int GT>
__device__ __forceinline__ void norm_group(const uint4 (*w)[Elem<GT>::kWords], int count, double &tot,
                                           uint32_t &bad)
{
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    uint32_t nz = 0;
#pragma unroll
    for (int k = 0; k < kNormVectors; ++k) {
        if (k < count) {
            bad |= Elem<GT>::nonfinite(w[k]);
            if constexpr (GT != ZERO_F16)
                nz |= Elem<GT>::nonzero(w[k]);
            float f[8];
            Elem<GT>::to_float(w[k], f);
#pragma unroll
            for (int e = 0; e < 8; ++e)
                acc[e] = __fmaf_rn(f[e], f[e], acc[e]);
        }
    }
    const float s = tree8(acc);
    if constexpr (GT == ZERO_F16) {
        tot += (double)s;
    } else if (s < __int_as_float(0x7F800000) && (s >= 0x1p-90f || nz == 0u)) {
        tot += (double)s;
    } else {
#pragma unroll
        for (int k = 0; k < kNormVectors; ++k) {
            if (k < count) {
                float f[8];
                Elem<GT>::to_float(w[k], f);
                tot += squares_wide(f);
            }
        }
    }
}

// 16-byte load that asks L2 to keep the line (evict-last priority).
__device__ __forceinline__ uint4 ld_keep(const uint4 *p)
{
    uint4 r;
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    asm volatile("ld.global.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p), "l"(pol));
    return r;
}

// Vectors [0, nv) of one array, thread `t` of `nt` taking vectors
// t, t + nt, ... kNormVectors at a time; then the scalar tail [8*nv, n).  Vectors
// from `keep_from` on are loaded with evict-last priority: pass 2 walks the
// shard from its end, so that tail of the gradient is still in L2 when pass
// 2 reads it again.
template <int GT>
__device__ __forceinline__ void norm_range(const void *g, int64_t n, int64_t t, int64_t nt, double &tot,
                                           uint32_t &bad, int64_t keep_from = INT64_MAX)
{
    constexpr int W = Elem<GT>::kWords;
    const uint4 *gv = static_cast<const uint4 *>(g);
    const int64_t nv = n >> 3;
    for (int64_t i = t; i < nv; i += kNormVectors * nt) {
        uint4 w[kNormVectors][W];
        int count = 0;
#pragma unroll
        for (int k = 0; k < kNormVectors; ++k) {
            const int64_t j = i + k * nt;
            if (j < nv) {
                if (j >= keep_from) {
#pragma unroll
                    for (int q = 0; q < W; ++q)
                        w[k][q] = ld_keep(gv + j * W + q);
                } else {
#pragma unroll
                    for (int q = 0; q < W; ++q)
                        w[k][q] = __ldcs(gv + j * W + q);
                }
                count = k + 1;
            }
        }
        norm_group<GT>(w, count, tot, bad);
    }
    const int64_t tail = n - (nv << 3);
    if (t < tail) {
        // the tail's squares in binary64 (any value of any type)
        const double x = Elem<GT>::scalar(g, (nv << 3) + t);
        bad |= Elem<GT>::scalar_nonfinite(g, (nv << 3) + t);
        tot += x * x;
    }
}

// The step decision, for a pass 1 whose last block takes it (a single-rank
// step: no cross-rank sum between the passes).
struct FoldedDecision {
    StepScalars *scp;     // NULL: pass 1 alone
    const PowCache *cache;
    DecideArgs a;
};

template <int GT>
__global__ void __launch_bounds__(kThreads, 4)
    k_norm_flat(const void *__restrict__ g, int64_t n, double2 *partials, WsHeader *hdr, zero_state_t *st,
                int accumulate, int trigger, FoldedDecision fd)
{
    if (trigger)
        pdl_launch_next();
    pdl_wait();
    double tot = 0.0;
    uint32_t bad = 0;
    // keep the last kL2KeepBytes of the gradient in L2 for pass 2
    const int64_t keep_vectors = kL2KeepBytes / (8 * Elem<GT>::kBytes);
    norm_range<GT>(g, n, (int64_t)blockIdx.x * kThreads + threadIdx.x, (int64_t)gridDim.x * kThreads, tot,
                   bad, (n >> 3) - keep_vectors);
    __shared__ DecideShared sh;
    if (norm_finish(tot, bad, partials, hdr, st, accumulate, &sh, fd.scp ? fd.cache : nullptr) && fd.scp) {
        // the last block, its totals in the state: the decision here saves
        // the decision kernel's launch and its dependency hop
        __syncthreads();
        decide_block(st, fd.scp, sh, fd.a);
    }
}

// Pass 1 over a large flat shard, the gradient staged through shared
// memory by bulk copies.  Each block holds a ring of kStages buffers of
// kStageBytes; one thread keeps the ring's chunks in flight, the block's
// threads read each chunk out of shared memory as it lands.  Block b takes
// the kStageBytes-chunks b, b + G, b + 2G, ... of the array (G blocks, two
// per SM).  Measured on GB300 over a binary16 gradient with L2 flushed:
// 455 us against 480 us for the register-loaded kernel at 1.56G elements,
// 94.9 against 98.9 us at 268M, level at 97M; the whole step 6.575 against
// 6.596 ms on the 1.56G shard and 0.4227 against 0.4249 ms on the 97.35M
// one.  Two blocks of three stages per SM measured best among one to four
// blocks of two to six stages: one block of eight warps per SM could not
// consume the chunks as fast as they landed (wait and barrier stalls), and
// deeper rings read more slowly.
constexpr int kStages = 3;
constexpr int kStageBytes = 16 << 10;
constexpr int kNormBulkBlocksPerSM = 2;
constexpr size_t kNormBulkSmem = (size_t)kStages * kStageBytes;
// Flat shards of at least this many whole chunks per SM, in plain device
// memory, take the staged kernel; smaller ones finish within a few memory
// round trips either way.
constexpr int64_t kBulkMinChunksPerSM = 8;
// A wait for a chunk gives up after this long (a copy that never lands);
// the block then reports the gradient as non-finite (the step is skipped)
// and counts the stall in the workspace header.
constexpr uint64_t kWaitLimitNs = 1000000000ull;

template <int GT>
__global__ void __launch_bounds__(kThreads, kNormBulkBlocksPerSM)
    k_norm_bulk(const void *__restrict__ g, int64_t n, double2 *partials, WsHeader *hdr, zero_state_t *st,
                int accumulate, int trigger, FoldedDecision fd, int64_t keep_chunk)
{
    extern __shared__ __align__(128) unsigned char ring[];
    __shared__ __align__(8) uint64_t full[kStages];
    if (trigger)
        pdl_launch_next();
    pdl_wait();
    constexpr int W = Elem<GT>::kWords;
    constexpr int kWordsPerThread = kStageBytes / 16 / kThreads;  // 4: 32 or 16 elements
    static_assert(kWordsPerThread % W == 0 && kWordsPerThread / W <= kNormVectors, "one norm group per chunk");
    const unsigned char *gb = static_cast<const unsigned char *>(g);
    const int64_t nch = n * Elem<GT>::kBytes / kStageBytes;
    const int64_t mine = (int64_t)blockIdx.x < nch ? (nch - 1 - blockIdx.x) / gridDim.x + 1 : 0;
    const uint64_t pol_keep = l2_policy(true), pol_stream = l2_policy(false);
    // chunk k of this block into buffer k mod kStages; the chunks of the
    // gradient's last kL2KeepBytes with evict-last priority (pass 2 starts
    // there)
    auto issue = [&](int64_t k) {
        const int64_t c = (int64_t)blockIdx.x + k * gridDim.x;
        const int s = (int)(k % kStages);
        bulk_load(ring + (size_t)s * kStageBytes, gb + c * kStageBytes, kStageBytes, &full[s],
                  c >= keep_chunk ? pol_keep : pol_stream);
    };
    if (threadIdx.x == 0) {
        mbar_init(full, kStages);
        for (int64_t k = 0; k < kStages && k < mine; ++k)
            issue(k);
    }
    __syncthreads();
    double tot = 0.0;
    uint32_t bad = 0;
    const uint64_t deadline = global_ns() + kWaitLimitNs;
    int64_t k = 0;
    for (; k < mine; ++k) {
        const int s = (int)(k % kStages);
        const bool ok = mbar_wait(&full[s], (uint32_t)((k / kStages) & 1), deadline);
        const uint4 *words = reinterpret_cast<const uint4 *>(ring + (size_t)s * kStageBytes);
        uint4 w[kWordsPerThread];
#pragma unroll
        for (int q = 0; q < kWordsPerThread; ++q)
            w[q] = words[q * kThreads + threadIdx.x];
        if (ok)
            norm_group<GT>(reinterpret_cast<const uint4(*)[W]>(w), kWordsPerThread / W, tot, bad);
        // every thread has read buffer s: it may be refilled
        if (!__syncthreads_and(ok))
            break;
        if (threadIdx.x == 0 && k + kStages < mine) {
            fence_proxy_async();
            issue(k + kStages);
        }
    }
    if (k < mine) {
        // a chunk did not land in time: report the gradient as non-finite,
        // count the stall, and let the copies still in flight land (with a
        // limit of their own) before the block's shared memory is released
        bad = 1;
        if (threadIdx.x == 0) {
            atomicAdd(&hdr->stalls, 1u);
            const uint64_t d2 = global_ns() + kWaitLimitNs;
            for (int64_t j = k; j < mine && j < k + kStages; ++j)
                mbar_wait(&full[j % kStages], (uint32_t)((j / kStages) & 1), d2);
        }
        __syncthreads();
    }
    // the elements after the last whole chunk (less than kStageBytes), by
    // the last block with plain loads
    if (blockIdx.x == gridDim.x - 1) {
        const int64_t first = nch * kStageBytes / Elem<GT>::kBytes;
        norm_range<GT>(gb + nch * kStageBytes, n - first, threadIdx.x, kThreads, tot, bad);
    }
    __shared__ DecideShared sh;
    if (norm_finish(tot, bad, partials, hdr, st, accumulate, &sh, fd.scp ? fd.cache : nullptr) && fd.scp) {
        __syncthreads();
        decide_block(st, fd.scp, sh, fd.a);
    }
}

template <int GT>
__global__ void __launch_bounds__(kThreads, 4)
    k_norm_list(const TensorEntry *__restrict__ ents, const WorkItem *__restrict__ chunks, int64_t n_chunks,
                double2 *partials, WsHeader *hdr, zero_state_t *st, int accumulate, int trigger, FoldedDecision fd)
{
    if (trigger)
        pdl_launch_next();
    pdl_wait();
    double tot = 0.0;
    uint32_t bad = 0;
    // a warp per work item: most tensors of a long list are far smaller than
    // a block's share, and eight warps hide eight items' table loads at once
    // (measured over 10,000 tensors against a block per 64 Ki-element item:
    // 1.300 against 1.319 ms per step; 8 Ki-element items balance the warps)
    const int lane = (int)(threadIdx.x & 31);
    for (int64_t c = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5); c < n_chunks;
         c += (int64_t)gridDim.x * kWarps) {
        const WorkItem ch = chunks[c];
        const TensorEntry e = ents[ch.tensor];
        const int64_t start = (int64_t)ch.index * kChunk;
        const int64_t len = min(kChunk, e.numel - start);
        const void *g = static_cast<const char *>(e.g) + start * Elem<GT>::kBytes;
        norm_range<GT>(g, len, lane, 32, tot, bad);
    }
    __shared__ DecideShared sh;
    if (norm_finish(tot, bad, partials, hdr, st, accumulate, &sh, fd.scp ? fd.cache : nullptr) && fd.scp) {
        // the last block, its totals in the state: the step decision here,
        // as over a flat shard
        __syncthreads();
        decide_block(st, fd.scp, sh, fd.a);
    }
}

// ------------------------------------------------------------- stage-2 reduction

// ZeRO stage 2 partitions the gradients: a rank keeps only the reduced
// gradient of its own shard ("ZeRO: Memory Optimizations Toward Training
// Trillion Parameter Models - 中文验证版", section 方法适配).  This kernel is the
// arithmetic of that reduction on one GPU -- the mean over the Nd replicas'
// slices of the shard, summed in rank order in binary32 and divided once --
// fused with pass 1 over the stored result.

constexpr int kMaxReplicas = 64;

struct ReplicaPtrs {
    const void *p[kMaxReplicas];
};

// Elements 8i .. 8i+7: the rank-ordered binary32 sum over the replicas,
// loading up to 8 replicas' vectors at a time.
template <int GT>
__device__ __forceinline__ void replica_sum(const ReplicaPtrs &r, int nr, int64_t i, float *a)
{
    constexpr int W = Elem<GT>::kWords;
    {
        uint4 w0[W];
#pragma unroll
        for (int q = 0; q < W; ++q)
            w0[q] = __ldcs(static_cast<const uint4 *>(r.p[0]) + i * W + q);
        Elem<GT>::to_float(w0, a);
    }
    for (int k0 = 1; k0 < nr; k0 += 8) {
        uint4 w[8][W];
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (k0 + j < nr) {
#pragma unroll
                for (int q = 0; q < W; ++q)
                    w[j][q] = __ldcs(static_cast<const uint4 *>(r.p[k0 + j]) + i * W + q);
            }
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (k0 + j < nr) {
                float f[8];
                Elem<GT>::to_float(w[j], f);
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    a[e] = __fadd_rn(a[e], f[e]);
            }
    }
}

// Stores 8 means as the output type; returns the stored values as binary32
// and their overflow bits.
template <int OT>
__device__ __forceinline__ uint32_t store_mean(void *out, int64_t i, const float *mean, float *stored)
{
    if constexpr (OT == ZERO_F32) {
        float4 *o = static_cast<float4 *>(out) + 2 * i;
        __stcs(o, make_float4(mean[0], mean[1], mean[2], mean[3]));
        __stcs(o + 1, make_float4(mean[4], mean[5], mean[6], mean[7]));
        uint4 w[2];
        w[0] = make_uint4(__float_as_uint(mean[0]), __float_as_uint(mean[1]), __float_as_uint(mean[2]),
                          __float_as_uint(mean[3]));
        w[1] = make_uint4(__float_as_uint(mean[4]), __float_as_uint(mean[5]), __float_as_uint(mean[6]),
                          __float_as_uint(mean[7]));
#pragma unroll
        for (int e = 0; e < 8; ++e)
            stored[e] = mean[e];
        return Elem<ZERO_F32>::nonfinite(w);
    } else {
        const uint4 packed = LowP<OT>::pack(mean);
        __stcs(static_cast<uint4 *>(out) + i, packed);
        Elem<OT>::to_float(&packed, stored);
        return Elem<OT>::nonfinite(&packed);
    }
}

template <int OT>
__device__ __forceinline__ float store_mean_scalar(void *out, int64_t j, float mean, uint32_t &bad)
{
    if constexpr (OT == ZERO_F32) {
        static_cast<float *>(out)[j] = mean;
        bad |= (__float_as_uint(mean) & 0x7F800000u) == 0x7F800000u;
        return mean;
    } else {
        LowP<OT>::store(out, j, mean);
        bad |= Elem<OT>::scalar_nonfinite(out, j);
        return Elem<OT>::scalar(out, j);
    }
}

// Vectors per thread of the stage-2 reduction's one-shot grid (measured best
// of 1, 2 and 4).
constexpr int kReduceVectors = 2;

// The reduction with pass 1 fused: one-shot grid, V vectors per thread, one
// partial per block and the two-level deterministic finish.  On GB300 this
// schedule streams 16 replicas at 6.9 TB/s where a persistent grid of 4
// blocks per SM reached 6.65 TB/s.
template <int GT, int OT, int V>
__global__ void __launch_bounds__(kThreads)
    k_reduce_norm(ReplicaPtrs r, int nr, void *__restrict__ out, int64_t n, double2 *block_partials,
                   GroupArea *ga, WsHeader *hdr, zero_state_t *st, int accumulate)
{
    pdl_wait();
    const float count = (float)nr;
    uint32_t bad = 0;
    const int64_t nv = n >> 3;
    const int64_t base = (int64_t)blockIdx.x * kThreads * V + threadIdx.x;
    float part = 0.0f;
    double wide = 0.0;  // squares of out-of-range vectors (bfloat16 / binary32 data)
#pragma unroll
    for (int u = 0; u < V; ++u) {
        const int64_t i = base + (int64_t)u * kThreads;
        if (i < nv) {
            float a[8], mean[8], stored[8];
            replica_sum<GT>(r, nr, i, a);
#pragma unroll
            for (int e = 0; e < 8; ++e)
                mean[e] = __fdiv_rn(a[e], count);
            bad |= store_mean<OT>(out, i, mean, stored);
            if constexpr (GT == ZERO_F16) {
                // means of binary16 values: every square is a normal binary32
                float sq[8];
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    sq[e] = __fmul_rn(stored[e], stored[e]);
                part = __fadd_rn(part, tree8(sq));
            } else {
                add_squares_checked(stored, nonzero8(stored), part, wide);
            }
        }
    }
    double tot = wide + (double)part;
    const int64_t tail = n - (nv << 3);
    if (blockIdx.x == 0 && threadIdx.x < tail) {
        const int64_t j = (nv << 3) + threadIdx.x;
        float a = Elem<GT>::scalar(r.p[0], j);
        for (int k = 1; k < nr; ++k)
            a = __fadd_rn(a, Elem<GT>::scalar(r.p[k], j));
        const double x = store_mean_scalar<OT>(out, j, __fdiv_rn(a, count), bad);
        tot += x * x;
    }
    uint32_t b = bad != 0;
    if (group_finish(tot, b, block_partials, ga, hdr))
        write_norm(st, tot, b, accumulate);
}

// ------------------------------------------------------------- pass 2

// One element of the AdamW update, binary32, every operation rounded to
// nearest on its own (no contraction):
//   g = (g_lp * inv_scale) * clip
//   m' = b1*m + omb1*g;   v' = b2*v + omb2*(g*g)
//   p' = p - (step_size * m' / (sqrt(v')*isb2 + eps) + lrwd*p)
__device__ __forceinline__ void adam_elem(float graw, float &p, float &m, float &v, const StepScalars &s)
{
    const float g = __fmul_rn(__fmul_rn(graw, s.inv_scale), s.clip);
    const float m1 = __fadd_rn(__fmul_rn(s.b1, m), __fmul_rn(s.omb1, g));
    const float v1 = __fadd_rn(__fmul_rn(s.b2, v), __fmul_rn(s.omb2, __fmul_rn(g, g)));
    const float d = __fadd_rn(__fmul_rn(__fsqrt_rn(v1), s.isb2), s.eps);
    const float u = __fdiv_rn(m1, d);
    p = __fsub_rn(p, __fadd_rn(__fmul_rn(s.step_size, u), __fmul_rn(s.lrwd, p)));
    m = m1;
    v = v1;
}

__device__ __forceinline__ void unpack8(const float4 &a, const float4 &b, float *f)
{
    f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
    f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
}

// 8 binary32 values at p: one 32-byte access (V32, p on a 32-byte boundary)
// or two 16-byte accesses, with streaming (evict-first) hints.  Over HBM the
// two are equally fast; over the host link (state in pinned host memory) the
// 32-byte form moves 2.4x more data per second.
template <bool V32>
__device__ __forceinline__ void ld8f(const float *p, float *f)
{
    if (V32) {
        asm("ld.global.cs.v8.f32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
            : "=f"(f[0]), "=f"(f[1]), "=f"(f[2]), "=f"(f[3]), "=f"(f[4]), "=f"(f[5]), "=f"(f[6]), "=f"(f[7])
            : "l"(p));
    } else {
        unpack8(__ldcs(reinterpret_cast<const float4 *>(p)), __ldcs(reinterpret_cast<const float4 *>(p) + 1), f);
    }
}

template <bool V32>
__device__ __forceinline__ void st8f(float *p, const float *f)
{
    if (V32) {
        asm volatile("st.global.cs.v8.f32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "f"(f[0]), "f"(f[1]),
                     "f"(f[2]), "f"(f[3]), "f"(f[4]), "f"(f[5]), "f"(f[6]), "f"(f[7])
                     : "memory");
    } else {
        __stcs(reinterpret_cast<float4 *>(p), make_float4(f[0], f[1], f[2], f[3]));
        __stcs(reinterpret_cast<float4 *>(p) + 1, make_float4(f[4], f[5], f[6], f[7]));
    }
}

// Vector i (elements 8i .. 8i+7) of one array set.
// The inputs of vector i (elements 8i .. 8i+7) of one array set.
template <int GT, bool V32>
__device__ __forceinline__ void adam_load(const void *g, const float *p, const float *m, const float *v, int64_t i,
                                          float *gf, float *pf, float *mf, float *vf)
{
    if (GT == ZERO_F32) {
        ld8f<V32>(static_cast<const float *>(g) + 8 * i, gf);
    } else {
        const uint4 gw = __ldcs(static_cast<const uint4 *>(g) + i);
        Elem<GT>::to_float(&gw, gf);
    }
    ld8f<V32>(p + 8 * i, pf);
    ld8f<V32>(m + 8 * i, mf);
    ld8f<V32>(v + 8 * i, vf);
}

// The update of vector i from its loaded inputs, and its stores.
template <int PT, bool V32>
__device__ __forceinline__ void adam_store(float *p, float *m, float *v, void *plp, int64_t i, const float *gf,
                                           float *pf, float *mf, float *vf, const StepScalars &s)
{
#pragma unroll
    for (int e = 0; e < 8; ++e)
        adam_elem(gf[e], pf[e], mf[e], vf[e], s);
    st8f<V32>(p + 8 * i, pf);
    st8f<V32>(m + 8 * i, mf);
    st8f<V32>(v + 8 * i, vf);
    if (plp)
        __stcs(static_cast<uint4 *>(plp) + i, LowP<PT>::pack(pf));
}

template <int GT, int PT, bool V32>
__device__ __forceinline__ void adam_vec(const void *g, float *p, float *m, float *v, void *plp, int64_t i,
                                         const StepScalars &s)
{
    float gf[8], pf[8], mf[8], vf[8];
    adam_load<GT, V32>(g, p, m, v, i, gf, pf, mf, vf);
    adam_store<PT, V32>(p, m, v, plp, i, gf, pf, mf, vf, s);
}

template <int GT, int PT>
__device__ __forceinline__ void adam_scalar(const void *g, float *p, float *m, float *v, void *plp, int64_t j,
                                            const StepScalars &s)
{
    float pj = p[j], mj = m[j], vj = v[j];
    adam_elem(Elem<GT>::scalar(g, j), pj, mj, vj, s);
    p[j] = pj;
    m[j] = mj;
    v[j] = vj;
    if (plp)
        LowP<PT>::store(plp, j, pj);
}

// One thread per 8-element vector, no loop: the grid covers the whole
// array once (ceil(n / 2048) blocks, taken from the end of the array), the
// last n mod 8 elements going to the threads just past the last vector.  Measured on GB300 this one-shot
// schedule streams the five arrays at about 7.0 TB/s where persistent
// grid-stride grids of 1 to 16 blocks per SM reach 5.1 to 6.8 TB/s.
template <int GT, int PT, bool V32>
__global__ void __launch_bounds__(kThreads, 4)
    k_adam_flat(const void *__restrict__ g, float *__restrict__ p, float *__restrict__ m, float *__restrict__ v,
                void *__restrict__ plp, int64_t n, const StepScalars *__restrict__ scp, PowCache *cache)
{
    const int64_t nv = n >> 3;
    // blocks walk the shard from its end: pass 1 left that end of the
    // gradient in L2
    const int64_t i = (int64_t)(gridDim.x - 1 - blockIdx.x) * kThreads + threadIdx.x;
    // the vector's inputs are loaded before the wait for the previous
    // kernel: that kernel (pass 1 or the decision, of the same call) writes
    // none of them, and it started only once all earlier work in the stream
    // had finished; so the blocks resident while it drains have their loads
    // in flight
    float gf[8], pf[8], mf[8], vf[8];
    if (i < nv)
        adam_load<GT, V32>(g, p, m, v, i, gf, pf, mf, vf);
    pdl_wait();
    const StepScalars s = load_scalars(scp);
    if (s.skip)
        return;
    if (i < nv)
        adam_store<PT, V32>(p, m, v, plp, i, gf, pf, mf, vf, s);
    else if (i - nv < (n & 7))
        adam_scalar<GT, PT>(g, p, m, v, plp, (nv << 3) + (i - nv), s);
    if (blockIdx.x == 0 && threadIdx.x < 32)
        refill_pow_window(s, cache);
}

// Pass 2 over a list: one block per tile of kTile elements of one tensor,
// kTileVectors vectors per thread (one-shot).  Two vectors (4096-element
// tiles) measured best over 10,000 tensors: 1.01 of the copy peak against
// 0.98 with one and 1.00 with four; each block first reads its work item and
// its tensor's entry, and larger tiles pay that once for more elements.
template <int GT, int PT, bool V32>
__global__ void __launch_bounds__(kThreads, 4)
    k_adam_list(const TensorEntry *__restrict__ ents, const WorkItem *__restrict__ tiles,
                const StepScalars *__restrict__ scp, PowCache *cache)
{
    pdl_wait();
    const StepScalars s = load_scalars(scp);
    if (s.skip)
        return;
    if (blockIdx.x == 0 && threadIdx.x < 32)
        refill_pow_window(s, cache);
    const WorkItem tl = tiles[blockIdx.x];
    const TensorEntry e = ents[tl.tensor];
    const int64_t start = (int64_t)tl.index * kTile;
    const int64_t len = min(kTile, e.numel - start);
    const void *g = static_cast<const char *>(e.g) + start * Elem<GT>::kBytes;
    void *plp = e.plp ? static_cast<void *>(static_cast<char *>(e.plp) + start * 2) : nullptr;
    const int64_t nv = len >> 3;
    const int64_t t = threadIdx.x;
#pragma unroll
    for (int u = 0; u < kTileVectors; ++u)
        if (t + u * kThreads < nv)
            adam_vec<GT, PT, V32>(g, e.p + start, e.m + start, e.v + start, plp, t + u * kThreads, s);
    // the tail of a tensor's last tile (up to 7 elements) goes to threads
    // 0..6, which may also hold a vector: nv + tail can exceed the block
    if (t < (len & 7))
        adam_scalar<GT, PT>(g, e.p + start, e.m + start, e.v + start, plp, (nv << 3) + t, s);
}

// ------------------------------------------------------------- accumulate

struct BufPtrs {
    const void *p[8];
};

template <int GT>
__global__ void __launch_bounds__(kThreads)
    k_accumulate(float *__restrict__ acc, BufPtrs b, int nb, int64_t n, int overwrite)
{
    constexpr int W = Elem<GT>::kWords;
    const int64_t nv = n >> 3;
    const int64_t nt = (int64_t)gridDim.x * kThreads;
    const int64_t t = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    for (int64_t i = t; i < nv; i += nt) {
        uint4 w[8][W];
#pragma unroll
        for (int k = 0; k < 8; ++k)
            if (k < nb) {
#pragma unroll
                for (int q = 0; q < W; ++q)
                    w[k][q] = __ldcs(static_cast<const uint4 *>(b.p[k]) + i * W + q);
            }
        float4 *a4 = reinterpret_cast<float4 *>(acc) + 2 * i;
        float a[8];
        int k0 = 0;
        if (overwrite) {
            Elem<GT>::to_float(w[0], a);
            k0 = 1;
        } else {
            unpack8(__ldcs(a4), __ldcs(a4 + 1), a);
        }
#pragma unroll
        for (int k = 0; k < 8; ++k)
            if (k >= k0 && k < nb) {
                float f[8];
                Elem<GT>::to_float(w[k], f);
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    a[e] = __fadd_rn(a[e], f[e]);
            }
        __stcs(a4, make_float4(a[0], a[1], a[2], a[3]));
        __stcs(a4 + 1, make_float4(a[4], a[5], a[6], a[7]));
    }
    const int64_t tail = n - (nv << 3);
    if (t < tail) {
        const int64_t j = (nv << 3) + t;
        float a = overwrite ? Elem<GT>::scalar(b.p[0], j) : acc[j];
#pragma unroll
        for (int k = 0; k < 8; ++k)
            if (k >= overwrite && k < nb)
                a = __fadd_rn(a, Elem<GT>::scalar(b.p[k], j));
        acc[j] = a;
    }
}

// ------------------------------------------------------------- accumulation with pass 1

// Gradient accumulation fused with pass 1: acc = (overwrite ? 0 : acc) +
// g_0 + ... + g_{nb-1} in binary32 in micro-batch order (as k_accumulate),
// stored, and the squared norm and overflow of the stored sums folded into
// the state (as pass 1 over acc would).  The fp32 sums are not read back:
// the step moves 4 bytes per element less than accumulation, then pass 1.
// Persistent grid with pass 1's finish (squares in binary32 lane sums over
// 4 vectors, one binary64 add per 32 elements, one ticket): a one-shot
// grid with the grouped finish measured 5.3 TB/s here, its per-block fence
// waiting behind 4 bytes per element of streaming stores.
template <int GT>
__global__ void __launch_bounds__(kThreads)
    k_accumulate_norm(float *__restrict__ acc, BufPtrs b, int nb, int64_t n, int overwrite, double2 *partials,
                      WsHeader *hdr, zero_state_t *st, int accumulate)
{
    constexpr int W = Elem<GT>::kWords;
    pdl_wait();
    uint32_t bad = 0;
    double tot = 0.0;
    float part = 0.0f;
    int groups = 0;
    const int64_t nv = n >> 3;
    const int64_t nt = (int64_t)gridDim.x * kThreads;
    const int64_t t = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    for (int64_t i = t; i < nv; i += nt) {
        uint4 w[8][W];
#pragma unroll
        for (int k = 0; k < 8; ++k)
            if (k < nb) {
#pragma unroll
                for (int q = 0; q < W; ++q)
                    w[k][q] = __ldcs(static_cast<const uint4 *>(b.p[k]) + i * W + q);
            }
        float a[8], stored[8];
        int k0 = 0;
        if (overwrite) {
            Elem<GT>::to_float(w[0], a);
            k0 = 1;
        } else {
            const float4 *a4 = reinterpret_cast<const float4 *>(acc) + 2 * i;
            unpack8(__ldcs(a4), __ldcs(a4 + 1), a);
        }
#pragma unroll
        for (int k = 0; k < 8; ++k)
            if (k >= k0 && k < nb) {
                float f[8];
                Elem<GT>::to_float(w[k], f);
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    a[e] = __fadd_rn(a[e], f[e]);
            }
        bad |= store_mean<ZERO_F32>(acc, i, a, stored);
        // binary32 sums (of any type, and of whatever acc held): squares
        // range-checked
        add_squares_checked(stored, nonzero8(stored), part, tot);
        if (++groups == 4) {
            tot += (double)part;
            part = 0.0f;
            groups = 0;
        }
    }
    tot += (double)part;
    const int64_t tail = n - (nv << 3);
    if (t < tail) {
        const int64_t j = (nv << 3) + t;
        float a = overwrite ? Elem<GT>::scalar(b.p[0], j) : acc[j];
#pragma unroll
        for (int k = 0; k < 8; ++k)
            if (k >= overwrite && k < nb)
                a = __fadd_rn(a, Elem<GT>::scalar(b.p[k], j));
        const double x = store_mean_scalar<ZERO_F32>(acc, j, a, bad);
        tot += x * x;
    }
    __shared__ DecideShared sh;
    norm_finish(tot, bad, partials, hdr, st, accumulate, &sh);
}

// A list's table as copied into the workspace.
struct ListDev {
    const TensorEntry *ents = nullptr;
    const WorkItem *tiles = nullptr;   // pass 2: one per kTile elements
    const WorkItem *chunks = nullptr;  // pass 1: one per kChunk elements
    int64_t n = 0, n_tiles = 0, n_chunks = 0;
    bool aligned32 = true;             // every fp32 array on 32 bytes
};

// Builds a list's table on the host -- one entry per tensor, then the work
// items of pass 2 and of pass 1 -- and copies it into the workspace in one
// stream-ordered copy.  p, m, v, plp may be NULL (pass 1 alone).  (Items
// indexed directly by block measured faster than a per-block search over
// per-tensor prefixes: 1.20 against 1.33 ms for pass 2 over 10,000 tensors.)
int upload_list(const zero_tlist_t *g, const zero_tlist_t *p, const zero_tlist_t *m, const zero_tlist_t *v,
                const zero_tlist_t *plp, void *ws, cudaStream_t stream, ListDev *L)
{
    const int64_t n = g->n;
    int64_t tiles = 0, chunks = 0;
    for (int64_t i = 0; i < n; ++i) {
        tiles += (g->numel[i] + kTile - 1) / kTile;
        chunks += (g->numel[i] + kChunk - 1) / kChunk;
    }
    if (tiles > 0x7fffffff)
        return ZERO_EINVAL;
    const size_t ent_bytes = align256((size_t)n * sizeof(TensorEntry));
    const size_t tile_bytes = align256((size_t)tiles * sizeof(WorkItem));
    std::vector<unsigned char> host(ent_bytes + tile_bytes + (size_t)chunks * sizeof(WorkItem));
    TensorEntry *ents = reinterpret_cast<TensorEntry *>(host.data());
    WorkItem *ti = reinterpret_cast<WorkItem *>(host.data() + ent_bytes);
    WorkItem *ch = reinterpret_cast<WorkItem *>(host.data() + ent_bytes + tile_bytes);
    bool a32 = true;
    int64_t t = 0, c = 0;
    for (int64_t i = 0; i < n; ++i) {
        TensorEntry &e = ents[i];
        e.g = g->ptrs[i];
        e.p = p ? static_cast<float *>(p->ptrs[i]) : nullptr;
        e.m = m ? static_cast<float *>(m->ptrs[i]) : nullptr;
        e.v = v ? static_cast<float *>(v->ptrs[i]) : nullptr;
        e.plp = plp ? plp->ptrs[i] : nullptr;
        e.numel = g->numel[i];
        if (p && e.numel > 0) {
            uintptr_t bits = reinterpret_cast<uintptr_t>(e.p) | reinterpret_cast<uintptr_t>(e.m) |
                             reinterpret_cast<uintptr_t>(e.v);
            if (g->dtype == ZERO_F32)
                bits |= reinterpret_cast<uintptr_t>(e.g);
            if (bits & 31u)
                a32 = false;
        }
        for (int64_t j = 0; j * kTile < e.numel; ++j)
            ti[t++] = WorkItem{(int32_t)i, (int32_t)j};
        for (int64_t j = 0; j * kChunk < e.numel; ++j)
            ch[c++] = WorkItem{(int32_t)i, (int32_t)j};
    }
    unsigned char *base = static_cast<unsigned char *>(ws) + kWsTable;
    if (!host.empty()) {
        const int rc = stage_upload(base, host.data(), host.size(), stream, "workspace table upload");
        if (rc != ZERO_OK)
            return rc;
    }
    L->ents = reinterpret_cast<const TensorEntry *>(base);
    L->tiles = reinterpret_cast<const WorkItem *>(base + ent_bytes);
    L->chunks = reinterpret_cast<const WorkItem *>(base + ent_bytes + tile_bytes);
    L->n = n;
    L->n_tiles = tiles;
    L->n_chunks = chunks;
    L->aligned32 = a32;
    return ZERO_OK;
}

// Pass 1.  `trigger`: the next operation in the stream is this library's
// decision kernel launched with PDL (the fused step), so the norm kernel may
// let it be scheduled early.
template <int GT>
int launch_norm(const zero_tlist_t *grads, int64_t total, zero_state_t *st, int accumulate, void *ws,
                cudaStream_t stream, bool trigger, const FoldedDecision &fd = FoldedDecision{},
                const ListDev *pre = nullptr)
{
    unsigned char *w = static_cast<unsigned char *>(ws);
    WsHeader *hdr = reinterpret_cast<WsHeader *>(w);
    double2 *partials = reinterpret_cast<double2 *>(w + kWsPartials);
    if (grads->n <= 1) {
        const void *g = grads->n == 1 ? grads->ptrs[0] : nullptr;
        const int64_t n = grads->n == 1 ? grads->numel[0] : 0;
        const int64_t chunks = n * Elem<GT>::kBytes / kStageBytes;
        const int sms = sm_count();
        if (sms > 0 && chunks >= kBulkMinChunksPerSM * sms && plain_device_ptr(g)) {
            // two blocks per SM, the gradient staged through shared memory
            const int64_t keep_chunk = chunks - kL2KeepBytes / kStageBytes;
            cudaFuncSetAttribute(k_norm_bulk<GT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kNormBulkSmem);
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3((unsigned)(sms * kNormBulkBlocksPerSM));
            cfg.blockDim = dim3((unsigned)kThreads);
            cfg.dynamicSmemBytes = kNormBulkSmem;
            cfg.stream = stream;
            cudaLaunchKernelEx(&cfg, k_norm_bulk<GT>, g, n, partials, hdr, st, accumulate, (int)trigger, fd,
                               keep_chunk);
            return check_launch("zero_grad_norm_overflow");
        }
        // persistent grid of 4 blocks per SM (measured best for this pass)
        const int64_t items = ((n >> 3) + 4 * kThreads - 1) / (4 * kThreads);
        const int grid = grid_for((const void *)k_norm_flat<GT>, items, kMaxBlocks, 4);
        launch_k(k_norm_flat<GT>, grid, kThreads, stream, false, g, n, partials, hdr, st, accumulate,
                 (int)trigger, fd);
        return check_launch("zero_grad_norm_overflow");
    }
    ListDev L;
    if (pre) {
        L = *pre;
    } else {
        const int rc = upload_list(grads, nullptr, nullptr, nullptr, nullptr, ws, stream, &L);
        if (rc != ZERO_OK)
            return rc;
    }
    const int grid = grid_for((const void *)k_norm_list<GT>, (L.n_chunks + kWarps - 1) / kWarps, kMaxBlocks, 4);
    launch_k(k_norm_list<GT>, grid, kThreads, stream, false, L.ents, L.chunks, L.n_chunks, partials, hdr, st,
             accumulate, (int)trigger, fd);
    (void)total;
    return check_launch("zero_grad_norm_overflow");
}

// Pass 2 (after the decision kernel, with PDL).  For a list the tile table
// was uploaded before the decision kernel (see run_step).  `aligned32`: every
// fp32 array starts on a 32-byte boundary, so the 32-byte access form runs.
template <int GT, int PT, bool V32>
int launch_adam_v(const zero_tlist_t *g, const zero_tlist_t *p, const zero_tlist_t *m, const zero_tlist_t *v,
                  const zero_tlist_t *plp, const StepScalars *sc, void *ws, cudaStream_t stream, const ListDev &L)
{
    PowCache *cache = reinterpret_cast<PowCache *>(static_cast<unsigned char *>(ws) + kWsPowCache);
    if (g->n == 1) {
        const int64_t n = g->numel[0];
        if (n == 0)
            return ZERO_OK;
        // one thread per 8-element vector plus the n mod 8 tail threads
        const int64_t threads = (n >> 3) + (n & 7);
        const int64_t grid = (threads + kThreads - 1) / kThreads;
        launch_k(k_adam_flat<GT, PT, V32>, (int)grid, kThreads, stream, true, (const void *)g->ptrs[0],
                 static_cast<float *>(p->ptrs[0]), static_cast<float *>(m->ptrs[0]),
                 static_cast<float *>(v->ptrs[0]), plp ? plp->ptrs[0] : nullptr, n, sc, cache);
        return check_launch("zero_adam_step");
    }
    if (L.n_tiles == 0)
        return ZERO_OK;
    // one-shot: one block per tile
    launch_k(k_adam_list<GT, PT, V32>, (int)L.n_tiles, kThreads, stream, true, L.ents, L.tiles, sc, cache);
    return check_launch("zero_adam_step");
}

template <int GT, int PT>
int launch_adam(const zero_tlist_t *g, const zero_tlist_t *p, const zero_tlist_t *m, const zero_tlist_t *v,
                const zero_tlist_t *plp, const StepScalars *sc, void *ws, cudaStream_t stream, const ListDev &L,
                bool aligned32)
{
    if (aligned32)
        return launch_adam_v<GT, PT, true>(g, p, m, v, plp, sc, ws, stream, L);
    return launch_adam_v<GT, PT, false>(g, p, m, v, plp, sc, ws, stream, L);
}

template <int GT>
int launch_adam_lp(int32_t pdtype, const zero_tlist_t *g, const zero_tlist_t *p, const zero_tlist_t *m,
                   const zero_tlist_t *v, const zero_tlist_t *plp, const StepScalars *sc, void *ws,
                   cudaStream_t stream, const ListDev &L, bool aligned32)
{
    if (pdtype == ZERO_BF16)
        return launch_adam<GT, ZERO_BF16>(g, p, m, v, plp, sc, ws, stream, L, aligned32);
    return launch_adam<GT, ZERO_F16>(g, p, m, v, plp, sc, ws, stream, L, aligned32);
}

// Checks the arguments of the decision + pass 2 part of a step.
// The state and hyper-parameter arguments of a step.
int check_state_hp(const zero_hparams_t *hp, zero_state_t *d_state)
{
    if (!hp || !d_state)
        return ZERO_EINVAL;
    if ((reinterpret_cast<uintptr_t>(d_state) & 7u) != 0)
        return ZERO_EALIGN;
    if (!device_ptr(d_state))
        return ZERO_EINVAL;
    if (!hparams_ok(hp))
        return ZERO_EINVAL;
    return ZERO_OK;
}

// The lists of a step and the workspace for them.
int check_lists(const zero_tlist_t *grads, const zero_tlist_t *master, const zero_tlist_t *m,
                const zero_tlist_t *v, const zero_tlist_t *p_lp, void *ws, size_t ws_bytes, int64_t *total)
{
    int64_t t2 = 0;
    int rc = check_list(grads, total);
    if (rc != ZERO_OK)
        return rc;
    // the fp32 state may live in pinned host memory (streamed over the
    // host link by pass 2: offload of the optimizer state)
    const zero_tlist_t *states[3] = {master, m, v};
    for (const zero_tlist_t *l : states) {
        if ((rc = check_list(l, &t2, true)) != ZERO_OK)
            return rc;
        if (l->dtype != ZERO_F32)
            return ZERO_EDTYPE;
        if ((rc = check_same_shape(grads, l)) != ZERO_OK)
            return rc;
    }
    if (p_lp) {
        if ((rc = check_list(p_lp, &t2)) != ZERO_OK)
            return rc;
        if (!lp_dtype_ok(p_lp->dtype))
            return ZERO_EDTYPE;
        if ((rc = check_same_shape(grads, p_lp)) != ZERO_OK)
            return rc;
    }
    if (!grad_dtype_ok(grads->dtype))
        return ZERO_EDTYPE;
    if (grads->n == 1 && ((grads->numel[0] >> 3) + 7) / kThreads >= 0x7fffffff)
        return ZERO_EINVAL;  // past 2^42 elements: beyond any device memory
    return check_ws(ws, ws_bytes, grads->n, *total);
}

int check_step_args(const zero_tlist_t *grads, const zero_tlist_t *master, const zero_tlist_t *m,
                    const zero_tlist_t *v, const zero_tlist_t *p_lp, const zero_hparams_t *hp,
                    zero_state_t *d_state, void *ws, size_t ws_bytes, int64_t *total)
{
    const int rc = check_state_hp(hp, d_state);
    return rc != ZERO_OK ? rc : check_lists(grads, master, m, v, p_lp, ws, ws_bytes, total);
}

// Pass 2 on checked arguments (after this call's decision).
int launch_pass2(const zero_tlist_t *grads, const zero_tlist_t *master, const zero_tlist_t *m,
                 const zero_tlist_t *v, const zero_tlist_t *p_lp, const StepScalars *sc, void *ws, cudaStream_t s,
                 const ListDev &L, bool aligned32)
{
    const int32_t pd = p_lp ? p_lp->dtype : ZERO_F16;
    switch (grads->dtype) {
    case ZERO_F16: return launch_adam_lp<ZERO_F16>(pd, grads, master, m, v, p_lp, sc, ws, s, L, aligned32);
    case ZERO_BF16: return launch_adam_lp<ZERO_BF16>(pd, grads, master, m, v, p_lp, sc, ws, s, L, aligned32);
    default: return launch_adam_lp<ZERO_F32>(pd, grads, master, m, v, p_lp, sc, ws, s, L, aligned32);
    }
}

// Every fp32 array of a one-array list (and an fp32 gradient) starts on a
// 32-byte boundary: pass 2 may use its 32-byte access form.
bool flat_aligned32(const zero_tlist_t *grads, const zero_tlist_t *master, const zero_tlist_t *m,
                    const zero_tlist_t *v)
{
    uintptr_t bits = reinterpret_cast<uintptr_t>(master->ptrs[0]) | reinterpret_cast<uintptr_t>(m->ptrs[0]) |
                     reinterpret_cast<uintptr_t>(v->ptrs[0]);
    if (grads->dtype == ZERO_F32)
        bits |= reinterpret_cast<uintptr_t>(grads->ptrs[0]);
    return (bits & 31u) == 0;
}

// The decision kernel and pass 2 on checked arguments.  A list's table is
// copied into the workspace first (unless `pre` says this call already did,
// before its pass 1), so that nothing but the decision kernel sits between
// that copy and pass 2.  `decide_pdl`: the previous operation in the stream
// is this library's pass-1 kernel of the same call.
int run_step(const zero_tlist_t *grads, const zero_tlist_t *master, const zero_tlist_t *m, const zero_tlist_t *v,
             const zero_tlist_t *p_lp, const zero_hparams_t *hp, zero_state_t *d_state, void *ws,
             cudaStream_t s, bool decide_pdl, const ListDev *pre = nullptr)
{
    int rc;
    ListDev L;
    bool aligned32 = grads->n != 1 || flat_aligned32(grads, master, m, v);
    if (grads->n > 1) {
        if (pre) {
            L = *pre;
        } else {
            if ((rc = upload_list(grads, master, m, v, p_lp, ws, s, &L)) != ZERO_OK)
                return rc;
            decide_pdl = false;  // a copy now precedes the decision kernel
        }
        aligned32 = L.aligned32;
    }
    StepScalars *sc = reinterpret_cast<StepScalars *>(static_cast<unsigned char *>(ws) + kWsScalars);
    const DecideArgs a = decide_args(hp);
    PowCache *cache = reinterpret_cast<PowCache *>(static_cast<unsigned char *>(ws) + kWsPowCache);
    launch_k(k_decide, 1, 64, s, decide_pdl, d_state, sc, cache, a, 0);
    if ((rc = check_launch("zero_adam_step (decision)")) != ZERO_OK)
        return rc;
    if (grads->n == 0)
        return ZERO_OK;
    return launch_pass2(grads, master, m, v, p_lp, sc, ws, s, L, aligned32);
}

}  // namespace
}  // namespace zpml

using namespace zpml;

extern "C" int zero_accumulate_grads(float *acc, const void *const *g, int32_t n_bufs, int32_t dtype,
                                     int64_t n, int32_t overwrite, void *stream)
{
    if (n < 0 || n_bufs < 1 || n_bufs > 8 || !g || (overwrite != 0 && overwrite != 1))
        return ZERO_EINVAL;
    if (!grad_dtype_ok(dtype))
        return ZERO_EDTYPE;
    if (n == 0)
        return ZERO_OK;
    if (!acc)
        return ZERO_EINVAL;
    if (!aligned16(acc))
        return ZERO_EALIGN;
    BufPtrs b = {};
    for (int k = 0; k < n_bufs; ++k) {
        if (!g[k])
            return ZERO_EINVAL;
        if (!aligned16(g[k]))
            return ZERO_EALIGN;
        b.p[k] = g[k];
    }
    if (!device_ptr(acc))
        return ZERO_EINVAL;
    for (int k = 0; k < n_bufs; ++k)
        if (!device_ptr(g[k]))
            return ZERO_EINVAL;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int64_t items = ((n >> 3) + kThreads - 1) / kThreads;
    switch (dtype) {
    case ZERO_F16: {
        const int grid = grid_for((const void *)k_accumulate<ZERO_F16>, items, 1 << 30);
        k_accumulate<ZERO_F16><<<grid, kThreads, 0, s>>>(acc, b, n_bufs, n, overwrite);
        break;
    }
    case ZERO_BF16: {
        const int grid = grid_for((const void *)k_accumulate<ZERO_BF16>, items, 1 << 30);
        k_accumulate<ZERO_BF16><<<grid, kThreads, 0, s>>>(acc, b, n_bufs, n, overwrite);
        break;
    }
    default: {
        const int grid = grid_for((const void *)k_accumulate<ZERO_F32>, items, 1 << 30);
        k_accumulate<ZERO_F32><<<grid, kThreads, 0, s>>>(acc, b, n_bufs, n, overwrite);
        break;
    }
    }
    return check_launch("zero_accumulate_grads");
}

namespace zpml {
namespace {
template <int GT>
int launch_accumulate_norm(float *acc, const BufPtrs &b, int nb, int64_t n, int overwrite, zero_state_t *st,
                           int accumulate, void *ws, cudaStream_t stream)
{
    unsigned char *w = static_cast<unsigned char *>(ws);
    // persistent: one partial per block in the norm partials (at most
    // kMaxBlocks blocks), the ticket in the header
    const int64_t items = ((n >> 3) + kThreads - 1) / kThreads;
    const int grid = grid_for((const void *)k_accumulate_norm<GT>, items, kMaxBlocks);
    launch_k(k_accumulate_norm<GT>, grid, kThreads, stream, false, acc, b, nb, n, overwrite,
             reinterpret_cast<double2 *>(w + kWsPartials), reinterpret_cast<WsHeader *>(w), st, accumulate);
    return check_launch("zero_accumulate_grads_norm");
}
}  // namespace
}  // namespace zpml

extern "C" int zero_accumulate_grads_norm(float *acc, const void *const *g, int32_t n_bufs, int32_t dtype,
                                          int64_t n, int32_t overwrite, zero_state_t *d_state, int32_t accumulate,
                                          void *ws, size_t ws_bytes, void *stream)
{
    if (n < 0 || n_bufs < 1 || n_bufs > 8 || !g || (overwrite != 0 && overwrite != 1) || !d_state ||
        (accumulate != 0 && accumulate != 1))
        return ZERO_EINVAL;
    if (!grad_dtype_ok(dtype))
        return ZERO_EDTYPE;
    if ((reinterpret_cast<uintptr_t>(d_state) & 7u) != 0)
        return ZERO_EALIGN;
    if (!device_ptr(d_state))
        return ZERO_EINVAL;
    BufPtrs b = {};
    if (n > 0) {
        if (!acc)
            return ZERO_EINVAL;
        if (!aligned16(acc))
            return ZERO_EALIGN;
        if (!device_ptr(acc))
            return ZERO_EINVAL;
        for (int k = 0; k < n_bufs; ++k) {
            if (!g[k])
                return ZERO_EINVAL;
            if (!aligned16(g[k]))
                return ZERO_EALIGN;
            if (!device_ptr(g[k]))
                return ZERO_EINVAL;
            b.p[k] = g[k];
        }
    }
    int rc = check_ws(ws, ws_bytes, 1, n);
    if (rc != ZERO_OK)
        return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    switch (dtype) {
    case ZERO_F16: return launch_accumulate_norm<ZERO_F16>(acc, b, n_bufs, n, overwrite, d_state, accumulate, ws, s);
    case ZERO_BF16: return launch_accumulate_norm<ZERO_BF16>(acc, b, n_bufs, n, overwrite, d_state, accumulate, ws, s);
    default: return launch_accumulate_norm<ZERO_F32>(acc, b, n_bufs, n, overwrite, d_state, accumulate, ws, s);
    }
}

namespace zpml {
namespace {
template <int GT, int OT>
int launch_reduce(const ReplicaPtrs &r, int nr, void *out, int64_t n, zero_state_t *st, int accumulate, void *ws,
                  cudaStream_t stream)
{
    unsigned char *w = static_cast<unsigned char *>(ws);
    WsHeader *hdr = reinterpret_cast<WsHeader *>(w);
    // one partial per block in the table region (which holds at least
    // n / 256 bytes: ceil(n / 4096) partials of 16 bytes), the group area
    // after the norm partials
    constexpr int V = kReduceVectors;
    const int64_t blocks = ((n >> 3) + (int64_t)kThreads * V - 1) / ((int64_t)kThreads * V);
    const int grid = blocks > 0 ? (int)blocks : 1;
    launch_k(k_reduce_norm<GT, OT, V>, grid, kThreads, stream, false, r, nr, out, n,
             reinterpret_cast<double2 *>(w + kWsTable), reinterpret_cast<GroupArea *>(w + kWsGroups), hdr, st,
             accumulate);
    return check_launch("zero_reduce_grads");
}

template <int GT>
int launch_reduce_ot(int32_t out_dtype, const ReplicaPtrs &r, int nr, void *out, int64_t n, zero_state_t *st,
                     int accumulate, void *ws, cudaStream_t stream)
{
    switch (out_dtype) {
    case ZERO_F16: return launch_reduce<GT, ZERO_F16>(r, nr, out, n, st, accumulate, ws, stream);
    case ZERO_BF16: return launch_reduce<GT, ZERO_BF16>(r, nr, out, n, st, accumulate, ws, stream);
    default: return launch_reduce<GT, ZERO_F32>(r, nr, out, n, st, accumulate, ws, stream);
    }
}
}  // namespace
}  // namespace zpml

extern "C" int zero_reduce_grads(const void *const *replicas, int32_t n_replicas, int32_t dtype, int64_t n,
                                 void *out, int32_t out_dtype, zero_state_t *d_state, int32_t accumulate,
                                 void *ws, size_t ws_bytes, void *stream)
{
    if (!replicas || n_replicas < 1 || n_replicas > kMaxReplicas || n < 0 || !d_state ||
        (accumulate != 0 && accumulate != 1))
        return ZERO_EINVAL;
    if ((n >> 3) / ((int64_t)kThreads * kReduceVectors) >= (int64_t)kGroupBlocks * kMaxGroups)
        return ZERO_ESIZE;  // past 2^34 elements: more blocks than the finish has groups for
    if (!grad_dtype_ok(dtype) || !grad_dtype_ok(out_dtype))
        return ZERO_EDTYPE;
    if ((reinterpret_cast<uintptr_t>(d_state) & 7u) != 0)
        return ZERO_EALIGN;
    if (!device_ptr(d_state))
        return ZERO_EINVAL;
    ReplicaPtrs r = {};
    if (n > 0) {
        if (!out)
            return ZERO_EINVAL;
        if (!aligned16(out))
            return ZERO_EALIGN;
        if (!device_ptr(out))
            return ZERO_EINVAL;
        for (int k = 0; k < n_replicas; ++k) {
            if (!replicas[k])
                return ZERO_EINVAL;
            if (!aligned16(replicas[k]))
                return ZERO_EALIGN;
            if (!device_ptr(replicas[k]))
                return ZERO_EINVAL;
            r.p[k] = replicas[k];
        }
    }
    int rc = check_ws(ws, ws_bytes, 1, n);
    if (rc != ZERO_OK)
        return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    switch (dtype) {
    case ZERO_F16: return launch_reduce_ot<ZERO_F16>(out_dtype, r, n_replicas, out, n, d_state, accumulate, ws, s);
    case ZERO_BF16: return launch_reduce_ot<ZERO_BF16>(out_dtype, r, n_replicas, out, n, d_state, accumulate, ws, s);
    default: return launch_reduce_ot<ZERO_F32>(out_dtype, r, n_replicas, out, n, d_state, accumulate, ws, s);
    }
}

extern "C" int zero_workspace_stalls(const void *ws, uint32_t *stalls, void *stream)
{
    if (!ws || !stalls)
        return ZERO_EINVAL;
    if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0)
        return ZERO_EALIGN;
    if (!device_ptr(ws))
        return ZERO_EINVAL;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const WsHeader *hdr = static_cast<const WsHeader *>(ws);
    unsigned int v = 0;
    cudaError_t e = cudaMemcpyAsync(&v, &hdr->stalls, sizeof v, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess)
        e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) {
        set_cuda_error("zero_workspace_stalls", (int)e, cudaGetErrorString(e));
        return ZERO_ECUDA;
    }
    *stalls = v;
    return ZERO_OK;
}

extern "C" int zero_grad_norm_overflow(const zero_tlist_t *grads, zero_state_t *d_state, int32_t accumulate,
                                       void *ws, size_t ws_bytes, void *stream)
{
    if (!d_state || (accumulate != 0 && accumulate != 1))
        return ZERO_EINVAL;
    if ((reinterpret_cast<uintptr_t>(d_state) & 7u) != 0)
        return ZERO_EALIGN;
    if (!device_ptr(d_state))
        return ZERO_EINVAL;
    int64_t total = 0;
    int rc = check_list(grads, &total);
    if (rc != ZERO_OK)
        return rc;
    if (!grad_dtype_ok(grads->dtype))
        return ZERO_EDTYPE;
    rc = check_ws(ws, ws_bytes, grads->n, total);
    if (rc != ZERO_OK)
        return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    switch (grads->dtype) {
    case ZERO_F16: return launch_norm<ZERO_F16>(grads, total, d_state, accumulate, ws, s, false);
    case ZERO_BF16: return launch_norm<ZERO_BF16>(grads, total, d_state, accumulate, ws, s, false);
    default: return launch_norm<ZERO_F32>(grads, total, d_state, accumulate, ws, s, false);
    }
}

extern "C" int zero_adam_step(const zero_tlist_t *grads, const zero_tlist_t *master, const zero_tlist_t *m,
                              const zero_tlist_t *v, const zero_tlist_t *p_lp, const zero_hparams_t *hp,
                              zero_state_t *d_state, void *ws, size_t ws_bytes, void *stream)
{
    int64_t total = 0;
    int rc = check_step_args(grads, master, m, v, p_lp, hp, d_state, ws, ws_bytes, &total);
    if (rc != ZERO_OK)
        return rc;
    // the caller's work (e.g. the cross-rank sum) may precede the decision
    // kernel: no early launch for it
    return run_step(grads, master, m, v, p_lp, hp, d_state, ws, static_cast<cudaStream_t>(stream), false);
}

// The step over a list whose table is in the workspace: pass 1 with the
// decision in its last block, then pass 2 (PDL) -- no decision kernel.
int list_step(const zero_tlist_t *grads, const zero_tlist_t *master, const zero_tlist_t *m, const zero_tlist_t *v,
              const zero_tlist_t *p_lp, const zero_hparams_t *hp, zero_state_t *d_state, void *ws, cudaStream_t s,
              const ListDev &L, int64_t total)
{
    unsigned char *w = static_cast<unsigned char *>(ws);
    StepScalars *sc = reinterpret_cast<StepScalars *>(w + kWsScalars);
    const FoldedDecision fd = {sc, reinterpret_cast<const PowCache *>(w + kWsPowCache), decide_args(hp)};
    int rc;
    switch (grads->dtype) {
    case ZERO_F16: rc = launch_norm<ZERO_F16>(grads, total, d_state, 0, ws, s, true, fd, &L); break;
    case ZERO_BF16: rc = launch_norm<ZERO_BF16>(grads, total, d_state, 0, ws, s, true, fd, &L); break;
    default: rc = launch_norm<ZERO_F32>(grads, total, d_state, 0, ws, s, true, fd, &L); break;
    }
    if (rc != ZERO_OK)
        return rc;
    return launch_pass2(grads, master, m, v, p_lp, sc, ws, s, L, L.aligned32);
}

extern "C" int zero_step(const zero_tlist_t *grads, const zero_tlist_t *master, const zero_tlist_t *m,
                         const zero_tlist_t *v, const zero_tlist_t *p_lp, const zero_hparams_t *hp,
                         zero_state_t *d_state, void *ws, size_t ws_bytes, void *stream)
{
    int64_t total = 0;
    int rc = check_step_args(grads, master, m, v, p_lp, hp, d_state, ws, ws_bytes, &total);
    if (rc != ZERO_OK)
        return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (grads->n == 1) {
        // a flat shard: the last block of pass 1 takes the decision, and
        // pass 2 follows with nothing in between (scheduled while pass 1
        // drains)
        unsigned char *w = static_cast<unsigned char *>(ws);
        StepScalars *sc = reinterpret_cast<StepScalars *>(w + kWsScalars);
        const FoldedDecision fd = {sc, reinterpret_cast<const PowCache *>(w + kWsPowCache), decide_args(hp)};
        switch (grads->dtype) {
        case ZERO_F16: rc = launch_norm<ZERO_F16>(grads, total, d_state, 0, ws, s, true, fd); break;
        case ZERO_BF16: rc = launch_norm<ZERO_BF16>(grads, total, d_state, 0, ws, s, true, fd); break;
        default: rc = launch_norm<ZERO_F32>(grads, total, d_state, 0, ws, s, true, fd); break;
        }
        if (rc != ZERO_OK)
            return rc;
        return launch_pass2(grads, master, m, v, p_lp, sc, ws, s, ListDev{}, flat_aligned32(grads, master, m, v));
    }
    if (grads->n == 0) {
        // nothing to update: pass 1 (an empty sum into the state), then the
        // decision kernel
        switch (grads->dtype) {
        case ZERO_F16: rc = launch_norm<ZERO_F16>(grads, total, d_state, 0, ws, s, false); break;
        case ZERO_BF16: rc = launch_norm<ZERO_BF16>(grads, total, d_state, 0, ws, s, false); break;
        default: rc = launch_norm<ZERO_F32>(grads, total, d_state, 0, ws, s, false); break;
        }
        if (rc != ZERO_OK)
            return rc;
        return run_step(grads, master, m, v, p_lp, hp, d_state, ws, s, false, nullptr);
    }
    // a list: its table copied once, for both passes, before pass 1; the
    // last block of pass 1 takes the decision and pass 2 follows, as over a
    // flat shard
    ListDev L;
    if ((rc = upload_list(grads, master, m, v, p_lp, ws, s, &L)) != ZERO_OK)
        return rc;
    return list_step(grads, master, m, v, p_lp, hp, d_state, ws, s, L, total);
}

// ------------------------------------------------------------- prepared steps

extern "C" int zero_list_prepare(const zero_tlist_t *grads, const zero_tlist_t *master, const zero_tlist_t *m,
                                 const zero_tlist_t *v, const zero_tlist_t *p_lp, void *ws, size_t ws_bytes,
                                 zero_list_plan_t *plan, void *stream)
{
    if (!plan)
        return ZERO_EINVAL;
    int64_t total = 0;
    int rc = check_lists(grads, master, m, v, p_lp, ws, ws_bytes, &total);
    if (rc != ZERO_OK)
        return rc;
    zero_list_plan_t P;
    std::memset(&P, 0, sizeof P);
    P.ws = ws;
    P.n = grads->n;
    P.total = total;
    P.gdtype = grads->dtype;
    P.pdtype = p_lp ? p_lp->dtype : -1;
    P.aligned32 = 1;
    if (grads->n == 1) {
        P.one[0] = grads->ptrs[0];
        P.one[1] = master->ptrs[0];
        P.one[2] = m->ptrs[0];
        P.one[3] = v->ptrs[0];
        P.one[4] = p_lp ? p_lp->ptrs[0] : nullptr;
    } else if (grads->n > 1) {
        ListDev L;
        if ((rc = upload_list(grads, master, m, v, p_lp, ws, static_cast<cudaStream_t>(stream), &L)) != ZERO_OK)
            return rc;
        P.ents = L.ents;
        P.tiles = L.tiles;
        P.chunks = L.chunks;
        P.n_tiles = L.n_tiles;
        P.n_chunks = L.n_chunks;
        P.aligned32 = L.aligned32 ? 1 : 0;
    }
    *plan = P;
    return ZERO_OK;
}

extern "C" int zero_step_prepared(const zero_list_plan_t *plan, const zero_hparams_t *hp, zero_state_t *d_state,
                                  void *ws, size_t ws_bytes, void *stream)
{
    if (!plan || plan->ws != ws || plan->n < 0 || !grad_dtype_ok(plan->gdtype) ||
        (plan->pdtype != -1 && !lp_dtype_ok(plan->pdtype)))
        return ZERO_EINVAL;
    int rc = check_state_hp(hp, d_state);
    if (rc != ZERO_OK)
        return rc;
    if ((rc = check_ws(ws, ws_bytes, plan->n, plan->total)) != ZERO_OK)
        return rc;
    if (plan->n <= 1) {
        // a one-array list (or none): zero_step on the pointers the plan holds
        void *g[1] = {plan->one[0]}, *p[1] = {plan->one[1]}, *mm[1] = {plan->one[2]}, *vv[1] = {plan->one[3]},
             *lp[1] = {plan->one[4]};
        const int64_t numel[1] = {plan->total};
        const zero_tlist_t tg = {g, numel, plan->n, plan->gdtype}, tp = {p, numel, plan->n, ZERO_F32},
                           tm = {mm, numel, plan->n, ZERO_F32}, tv = {vv, numel, plan->n, ZERO_F32},
                           tl = {lp, numel, plan->n, plan->pdtype};
        return zero_step(&tg, &tp, &tm, &tv, plan->pdtype >= 0 ? &tl : nullptr, hp, d_state, ws, ws_bytes, stream);
    }
    // the lists as far as the launches read them (their count and types);
    // every array pointer comes from the resident table
    const zero_tlist_t tg = {nullptr, nullptr, plan->n, plan->gdtype}, tf = {nullptr, nullptr, plan->n, ZERO_F32},
                       tl = {nullptr, nullptr, plan->n, plan->pdtype};
    ListDev L;
    L.ents = static_cast<const TensorEntry *>(plan->ents);
    L.tiles = static_cast<const WorkItem *>(plan->tiles);
    L.chunks = static_cast<const WorkItem *>(plan->chunks);
    L.n = plan->n;
    L.n_tiles = plan->n_tiles;
    L.n_chunks = plan->n_chunks;
    L.aligned32 = plan->aligned32 != 0;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return list_step(&tg, &tf, &tf, &tf, plan->pdtype >= 0 ? &tl : nullptr, hp, d_state, ws, s, L, plan->total);
}

// ------------------------------------------------------------- pass 1 without workspace
//
// A variant of pass 1 for callers that cannot hand the library a device
// workspace, because they cannot allocate device memory themselves: code that
// runs where another component owns all device memory (a training framework
// whose caching allocator has reserved the GPU, a plugin host that gives a
// plugin only its input and output buffers), or code that must keep the
// memory footprint of the step fixed.  Its scratch (the reduction ticket and
// the per-block partials) lives in one file-scope device array that every
// GPU loading this library holds until the process exits.

namespace zpml {
namespace {

constexpr int kStaticMaxArrays = 32;   // arrays per call
constexpr int kStaticMaxBlocks = 1024; // grid cap: one binary64 partial pair per block
constexpr size_t kStaticScratchBytes = 256 + 16 * (size_t)kStaticMaxBlocks;

static __device__ __align__(256) unsigned char g_norm_scratch[kStaticScratchBytes];

struct StaticArrays {
    const void *g[kStaticMaxArrays];
    int64_t n[kStaticMaxArrays];
};

template <int GT>
__global__ void __launch_bounds__(kThreads)
    k_norm_static(StaticArrays a, int n_arrays, unsigned char *scratch, zero_state_t *st, int accumulate)
{
    WsHeader *hdr = reinterpret_cast<WsHeader *>(scratch);
    double2 *partials = reinterpret_cast<double2 *>(scratch + 256);
    double tot = 0.0;
    uint32_t bad = 0;
    const int64_t t = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    const int64_t nt = (int64_t)gridDim.x * kThreads;
    for (int k = 0; k < n_arrays; ++k)
        norm_range<GT>(a.g[k], a.n[k], t, nt, tot, bad);
    __shared__ DecideShared sh;
    norm_finish(tot, bad, partials, hdr, st, accumulate, &sh);
}

// The identity of the calling thread's current context (cuCtxGetId, reached
// through the runtime's driver entry points, so the library does not link
// the driver library itself); 0 if it cannot be had.  A device reset
// (cudaDeviceReset) destroys the context and this library's module with it;
// the next context gets a new identity and the module a new load.
unsigned long long current_context_id()
{
    static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
    static PFN_cuCtxGetId_v12000 get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 4000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(f);
        f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(f);
        cudaGetLastError();
    });
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

// Device address of g_norm_scratch in the current context.  Looked up with
// cudaGetSymbolAddress (the device current) the first time a device is used
// and cached per device together with the context's identity; looked up
// again when that identity changes (after a device reset) or cannot be had.
// NULL on failure.
void *static_scratch()
{
    struct Entry {
        unsigned long long ctx = 0;
        void *addr = nullptr;
    };
    static std::mutex mu;
    static Entry cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        cudaGetLastError();
        return nullptr;
    }
    // the context exists once the caller's tensors do; this call makes sure
    const unsigned long long ctx = current_context_id();
    std::lock_guard<std::mutex> lock(mu);
    Entry &e = cache[dev];
    if (!e.addr || ctx == 0 || e.ctx != ctx) {
        void *p = nullptr;
        const cudaError_t err = cudaGetSymbolAddress(&p, g_norm_scratch);
        if (err != cudaSuccess) {
            set_cuda_error("zero_grad_norm_overflow_static (scratch address)", (int)err, cudaGetErrorString(err));
            cudaGetLastError();
            e = Entry{};
            return nullptr;
        }
        e.addr = p;
        e.ctx = ctx;
    }
    return e.addr;
}

template <int GT>
int launch_norm_static(const zero_tlist_t *grads, int64_t total, zero_state_t *st, int accumulate,
                       unsigned char *scratch, cudaStream_t stream)
{
    StaticArrays a = {};
    for (int64_t i = 0; i < grads->n; ++i) {
        a.g[i] = grads->ptrs[i];
        a.n[i] = grads->numel[i];
    }
    const int64_t items = ((total >> 3) + 4 * kThreads - 1) / (4 * kThreads);
    const int grid = grid_for((const void *)k_norm_static<GT>, items, kStaticMaxBlocks);
    k_norm_static<GT><<<grid, kThreads, 0, stream>>>(a, (int)grads->n, scratch, st, accumulate);
    return check_launch("zero_grad_norm_overflow_static");
}

}  // namespace
}  // namespace zpml

extern "C" int zero_grad_norm_overflow_static(const zero_tlist_t *grads, zero_state_t *d_state,
                                              int32_t accumulate, void *stream)
{
    if (!d_state || (accumulate != 0 && accumulate != 1))
        return ZERO_EINVAL;
    if ((reinterpret_cast<uintptr_t>(d_state) & 7u) != 0)
        return ZERO_EALIGN;
    if (!device_ptr(d_state))
        return ZERO_EINVAL;
    int64_t total = 0;
    int rc = check_list(grads, &total);
    if (rc != ZERO_OK)
        return rc;
    if (!grad_dtype_ok(grads->dtype))
        return ZERO_EDTYPE;
    if (grads->n > kStaticMaxArrays)
        return ZERO_ECAPACITY;
    unsigned char *scratch = static_cast<unsigned char *>(static_scratch());
    if (!scratch)
        return ZERO_ECUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // the ticket must start at zero whatever an earlier call left behind
    if (cudaMemsetAsync(scratch, 0, 256, s) != cudaSuccess)
        return check_launch("zero_grad_norm_overflow_static (ticket reset)");
    switch (grads->dtype) {
    case ZERO_F16: return launch_norm_static<ZERO_F16>(grads, total, d_state, accumulate, scratch, s);
    case ZERO_BF16: return launch_norm_static<ZERO_BF16>(grads, total, d_state, accumulate, scratch, s);
    default: return launch_norm_static<ZERO_F32>(grads, total, d_state, accumulate, scratch, s);
    }
}
