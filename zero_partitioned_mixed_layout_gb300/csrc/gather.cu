// ZeRO stage 3 on one GPU: the parameter gather (shards -> tensors) and its
// inverse (tensors -> shards).
//
// Source: "ZeRO: Memory Optimizations Toward Training Trillion Parameter
// Models - 中文验证版" (ai-papers.xuzou.cn), section 方法适配: stage 3
// partitions the parameters over the data-parallel ranks as well, so a rank
// assembles a tensor (or a layer) from all ranks' shards before using it.
// The flat buffer is the rank-order concatenation of the Nd shards, and
// tensor i is its slice [offset_i, offset_i + numel_i).
//
// The work is a copy, bound by HBM: 2 x element size bytes per element.  The
// kernel runs one block per 32 KiB tile of a tensor (one-shot grid, as the
// streaming passes of the optimizer step do), finds its tensor by a binary
// search over the tile prefix of the entry table, and splits the tile where
// it crosses a shard boundary.  Each span is copied with 16-byte stores; when
// source and destination differ in their offset modulo 16 bytes, each store
// is assembled from two 16-byte source loads with funnel shifts.
#include <algorithm>
#include <cstdint>
#include <vector>

#include "common.cuh"

namespace zpml {
namespace {

// 16-byte vectors per thread in one tile, and the tile size in bytes.  32 KiB
// tiles measured best on GB300 for the GPT-2 gather: 1.02 of the copy peak
// against 0.94 with 16 KiB and 0.98 with 64 KiB (the block's entry search
// and span set-up are paid once per tile).  At 4 blocks per SM the
// misaligned path, with two source granules per vector, spills 40-48 bytes
// to the stack; 3 blocks per SM (74 registers, no spill) measured 1.3 %
// slower on the aligned copies that dominate.
constexpr int kCopyVec = 8;
constexpr int64_t kCopyTile = (int64_t)kThreads * kCopyVec * 16;

// One tensor of the call: its device array, its size and flat position in
// bytes, and the index of its first tile.
struct GatherEntry {
    char *ptr;
    int64_t bytes;
    int64_t flat;
    int64_t tile0;
};

__device__ __forceinline__ uint4 ld_stream(const char *p)
{
    return __ldcs(reinterpret_cast<const uint4 *>(p));
}

__device__ __forceinline__ uint4 ld_cached(const char *p)
{
    return __ldg(reinterpret_cast<const uint4 *>(p));
}

__device__ __forceinline__ void st_stream(char *p, uint4 v) { __stcs(reinterpret_cast<uint4 *>(p), v); }

// The 16 bytes starting `k` bytes into the 32 bytes a:b (k in 0..15; k is a
// multiple of the element size, and uniform across the block).
__device__ __forceinline__ uint4 shifted(const uint4 &a, const uint4 &b, int k)
{
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    const int sh = (k & 3) * 8;
    uint4 o;
    switch (k >> 2) {
    case 0:
        o = make_uint4(__funnelshift_r(w[0], w[1], sh), __funnelshift_r(w[1], w[2], sh),
                       __funnelshift_r(w[2], w[3], sh), __funnelshift_r(w[3], w[4], sh));
        break;
    case 1:
        o = make_uint4(__funnelshift_r(w[1], w[2], sh), __funnelshift_r(w[2], w[3], sh),
                       __funnelshift_r(w[3], w[4], sh), __funnelshift_r(w[4], w[5], sh));
        break;
    case 2:
        o = make_uint4(__funnelshift_r(w[2], w[3], sh), __funnelshift_r(w[3], w[4], sh),
                       __funnelshift_r(w[4], w[5], sh), __funnelshift_r(w[5], w[6], sh));
        break;
    default:
        o = make_uint4(__funnelshift_r(w[3], w[4], sh), __funnelshift_r(w[4], w[5], sh),
                       __funnelshift_r(w[5], w[6], sh), __funnelshift_r(w[6], w[7], sh));
        break;
    }
    return o;
}

template <int ES>
__device__ __forceinline__ void copy_elem(char *dst, const char *src)
{
    if (ES == 2)
        *reinterpret_cast<uint16_t *>(dst) = *reinterpret_cast<const uint16_t *>(src);
    else
        *reinterpret_cast<uint32_t *>(dst) = *reinterpret_cast<const uint32_t *>(src);
}

// The whole block copies `len` bytes from src to dst (both multiples of ES
// bytes from a 16-byte boundary; len a multiple of ES).  Every load stays
// inside [src, src + len).
template <int ES>
__device__ __forceinline__ void copy_span(char *dst, const char *src, int64_t len)
{
    const int64_t d0 = (int64_t)reinterpret_cast<uintptr_t>(dst);
    const int64_t s0 = (int64_t)reinterpret_cast<uintptr_t>(src);
    const int k = (int)((s0 - d0) & 15);
    // Destination vectors D (16-byte aligned) whose source bytes lie in
    // 16-byte granules inside the span: D >= d0 + k, and D + 16 (+ 16 - k
    // when the source is shifted) <= d0 + len.
    const int64_t vlo = (d0 + k + 15) & ~(int64_t)15;
    const int64_t last = d0 + len - 16 - (k ? 16 - k : 0);
    const int64_t nv = last >= vlo ? ((last & ~(int64_t)15) - vlo) / 16 + 1 : 0;
    const int64_t body0 = nv ? vlo - d0 : len, body1 = nv ? vlo + 16 * nv - d0 : len;
    const int tid = threadIdx.x;

    for (int64_t base = 0; base < nv; base += (int64_t)kThreads * kCopyVec) {
        uint4 a[kCopyVec] = {}, b[kCopyVec] = {};
        if (k == 0) {
#pragma unroll
            for (int u = 0; u < kCopyVec; ++u) {
                const int64_t j = base + tid + u * kThreads;
                if (j < nv)
                    a[u] = ld_stream(src + (vlo - d0) + 16 * j);
            }
        } else {
#pragma unroll
            for (int u = 0; u < kCopyVec; ++u) {
                const int64_t j = base + tid + u * kThreads;
                if (j < nv) {
                    // the granule holding the vector's first source byte, and the next
                    const char *g = src + (vlo - d0) + 16 * j - k;
                    a[u] = ld_cached(g);
                    b[u] = ld_cached(g + 16);
                }
            }
#pragma unroll
            for (int u = 0; u < kCopyVec; ++u)
                a[u] = shifted(a[u], b[u], k);
        }
#pragma unroll
        for (int u = 0; u < kCopyVec; ++u) {
            const int64_t j = base + tid + u * kThreads;
            if (j < nv)
                st_stream(dst + (vlo - d0) + 16 * j, a[u]);
        }
    }
    // Head [0, body0) and tail [body1, len), element by element.
    const int64_t head = body0 / ES, tail = (len - body1) / ES;
    for (int64_t e = tid; e < head + tail; e += kThreads) {
        const int64_t off = e < head ? e * ES : body1 + (e - head) * ES;
        copy_elem<ES>(dst + off, src + off);
    }
}

// One block per tile: finds its tensor, then copies the tile's spans.
// kGather: shards -> tensors; else tensors -> shards.
template <bool kGather, int ES>
__device__ __forceinline__ void gather_tile(const GatherEntry *ents, int64_t n_ents, char *const *shards,
                                            int64_t shard_bytes)
{
    const int64_t tile = blockIdx.x;
    int64_t lo = 0, hi = n_ents - 1;
    while (lo < hi) {
        const int64_t mid = (lo + hi + 1) >> 1;
        if (ents[mid].tile0 <= tile)
            lo = mid;
        else
            hi = mid - 1;
    }
    const GatherEntry e = ents[lo];
    int64_t b = (tile - e.tile0) * kCopyTile;
    const int64_t b1 = b + kCopyTile < e.bytes ? b + kCopyTile : e.bytes;
    while (b < b1) {
        const int64_t f = e.flat + b;
        const int64_t r = f / shard_bytes;
        const int64_t in_shard = f - r * shard_bytes;
        const int64_t len = b1 - b < shard_bytes - in_shard ? b1 - b : shard_bytes - in_shard;
        char *t = e.ptr + b;
        char *s = shards[r] + in_shard;
        if (kGather)
            copy_span<ES>(t, s, len);
        else
            copy_span<ES>(s, t, len);
        b += len;
    }
}

// The tables in device memory (the workspace).
template <bool kGather, int ES>
__global__ void __launch_bounds__(kThreads, 4) k_gather(const GatherEntry *__restrict__ ents, int64_t n_ents,
                                                     char *const *__restrict__ shards, int64_t shard_bytes)
{
    gather_tile<kGather, ES>(ents, n_ents, shards, shard_bytes);
}

// Small calls (a layer of the per-layer schedule, a few tensors): the
// tables travel in the kernel's argument block, so the call uploads nothing
// before its launch.
constexpr int kArgEntries = 64;
constexpr int kArgShards = 256;
struct GatherArgs {
    GatherEntry ents[kArgEntries];
    char *shards[kArgShards];
};

template <bool kGather, int ES>
__global__ void __launch_bounds__(kThreads, 4) k_gather_args(const __grid_constant__ GatherArgs a, int64_t n_ents,
                                                          int64_t shard_bytes)
{
    gather_tile<kGather, ES>(a.ents, n_ents, a.shards, shard_bytes);
}

// ------------------------------------------------------------- host side

size_t entries_bytes(int64_t n) { return align256((size_t)(n > 0 ? n : 1) * sizeof(GatherEntry)); }
size_t shard_table_bytes(int32_t nd) { return align256((size_t)(nd > 0 ? nd : 1) * sizeof(char *)); }

int run_copy(bool gather, void *const *shards, int32_t nd, int64_t shard_numel, const zero_tlist_t *tl,
             const int64_t *offs, void *ws, size_t ws_bytes, void *stream)
{
    if (!tl || nd < 1 || shard_numel < 0 || !shards || tl->n < 0 || (tl->n > 0 && (!tl->ptrs || !tl->numel || !offs)))
        return ZERO_EINVAL;
    if (tl->dtype != ZERO_F16 && tl->dtype != ZERO_BF16 && tl->dtype != ZERO_F32)
        return ZERO_EDTYPE;
    const int es = tl->dtype == ZERO_F32 ? 4 : 2;
    const int64_t kLimit = (int64_t)1 << 62;
    if (shard_numel > kLimit / nd / es)
        return ZERO_ELAYOUT;
    const int64_t flat_total = shard_numel * nd;
    for (int32_t r = 0; r < nd; ++r) {
        if (!shards[r])
            return ZERO_EINVAL;
        if (!aligned16(shards[r]))
            return ZERO_EALIGN;
    }
    // Entries in list order, empty tensors dropped.
    std::vector<GatherEntry> ents;
    ents.reserve((size_t)tl->n);
    std::vector<std::pair<int64_t, int64_t>> ranges;
    int64_t tiles = 0;
    for (int64_t i = 0; i < tl->n; ++i) {
        const int64_t n = tl->numel[i], o = offs[i];
        if (n < 0 || o < 0)
            return ZERO_EINVAL;
        if (n == 0)
            continue;
        if (!tl->ptrs[i])
            return ZERO_EINVAL;
        if (!aligned16(tl->ptrs[i]))
            return ZERO_EALIGN;
        if (o > flat_total || n > flat_total - o)
            return ZERO_ELAYOUT;
        ents.push_back({static_cast<char *>(tl->ptrs[i]), n * es, o * es, tiles});
        tiles += (n * es + kCopyTile - 1) / kCopyTile;
        if (!gather)
            ranges.push_back({o, o + n});
    }
    if (!gather && ranges.size() > 1) {
        std::sort(ranges.begin(), ranges.end());
        for (size_t i = 1; i < ranges.size(); ++i)
            if (ranges[i].first < ranges[i - 1].second)
                return ZERO_ELAYOUT;
    }
    if (!ws)
        return ZERO_EWORKSPACE;
    if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0)
        return ZERO_EALIGN;
    if (ws_bytes < zero_gather_workspace_bytes(tl->n, nd))
        return ZERO_EWORKSPACE;
    if (!device_ptr(ws) || !device_ptr(shards[0]) || !device_ptr(shards[nd - 1]))
        return ZERO_EINVAL;
    if (!ents.empty() && (!device_ptr(ents.front().ptr) || !device_ptr(ents.back().ptr)))
        return ZERO_EINVAL;
    if (ents.empty())
        return ZERO_OK;
    if (tiles > 0x7fffffff)
        return ZERO_ELAYOUT;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int64_t n_ents = (int64_t)ents.size(), shard_bytes = shard_numel * es;
    const dim3 grid((unsigned)tiles), block(kThreads);
    if (n_ents <= kArgEntries && nd <= kArgShards) {
        GatherArgs a;
        std::copy(ents.begin(), ents.end(), a.ents);
        for (int32_t r = 0; r < nd; ++r)
            a.shards[r] = static_cast<char *>(shards[r]);
        if (gather && es == 2)
            k_gather_args<true, 2><<<grid, block, 0, st>>>(a, n_ents, shard_bytes);
        else if (gather)
            k_gather_args<true, 4><<<grid, block, 0, st>>>(a, n_ents, shard_bytes);
        else if (es == 2)
            k_gather_args<false, 2><<<grid, block, 0, st>>>(a, n_ents, shard_bytes);
        else
            k_gather_args<false, 4><<<grid, block, 0, st>>>(a, n_ents, shard_bytes);
        return check_launch(gather ? "k_gather (gather)" : "k_gather (scatter)");
    }

    // Tables: the shard pointers, then the entries.
    const size_t sb = shard_table_bytes(nd);
    std::vector<unsigned char> host(sb + ents.size() * sizeof(GatherEntry));
    std::copy(shards, shards + nd, reinterpret_cast<void **>(host.data()));
    std::copy(ents.begin(), ents.end(), reinterpret_cast<GatherEntry *>(host.data() + sb));
    unsigned char *base = static_cast<unsigned char *>(ws);
    const int rc = stage_upload(base, host.data(), host.size(), st, "gather table upload");
    if (rc != ZERO_OK)
        return rc;
    char *const *d_shards = reinterpret_cast<char *const *>(base);
    const GatherEntry *d_ents = reinterpret_cast<const GatherEntry *>(base + sb);
    if (gather && es == 2)
        k_gather<true, 2><<<grid, block, 0, st>>>(d_ents, n_ents, d_shards, shard_bytes);
    else if (gather)
        k_gather<true, 4><<<grid, block, 0, st>>>(d_ents, n_ents, d_shards, shard_bytes);
    else if (es == 2)
        k_gather<false, 2><<<grid, block, 0, st>>>(d_ents, n_ents, d_shards, shard_bytes);
    else
        k_gather<false, 4><<<grid, block, 0, st>>>(d_ents, n_ents, d_shards, shard_bytes);
    return check_launch(gather ? "k_gather (gather)" : "k_gather (scatter)");
}

}  // namespace
}  // namespace zpml

using namespace zpml;

extern "C" size_t zero_gather_workspace_bytes(int64_t n_tensors, int32_t nd)
{
    return shard_table_bytes(nd) + entries_bytes(n_tensors);
}

extern "C" int zero_gather_params(const void *const *shards, int32_t nd, int64_t shard_numel,
                                  const zero_tlist_t *tensors, const int64_t *tensor_offset, void *ws,
                                  size_t ws_bytes, void *stream)
{
    return run_copy(true, const_cast<void *const *>(shards), nd, shard_numel, tensors, tensor_offset, ws, ws_bytes,
                    stream);
}

extern "C" int zero_scatter_params(const zero_tlist_t *tensors, const int64_t *tensor_offset, void *const *shards,
                                   int32_t nd, int64_t shard_numel, void *ws, size_t ws_bytes, void *stream)
{
    return run_copy(false, shards, nd, shard_numel, tensors, tensor_offset, ws, ws_bytes, stream);
}
