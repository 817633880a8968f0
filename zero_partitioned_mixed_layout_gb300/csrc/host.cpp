// Host-only entry points of the C ABI: error strings, the flat partition
// layout, the stage-3 per-layer gather plan, the initial optimizer state and
// the workspace sizes.
//
// Layout source: "ZeRO: Memory Optimizations Toward Training Trillion
// Parameter Models - 中文验证版" (ai-papers.xuzou.cn), section 方法适配
// (method): ZeRO splits the model states (optimizer state, gradients,
// parameters) across the data-parallel ranks instead of replicating them.
#include <cmath>
#include <cstdio>
#include <cstring>
#include <vector>

#include "zero_pml_internal.h"

namespace zpml {

static thread_local char g_err[512];

void set_cuda_error(const char *what, int cuda_code, const char *cuda_msg)
{
    std::snprintf(g_err, sizeof g_err, "CUDA error %d (%s) in %s", cuda_code,
                  cuda_msg ? cuda_msg : "?", what ? what : "?");
}

}  // namespace zpml

extern "C" const char *zero_strerror(int code)
{
    static thread_local char buf[640];
    const char *base;
    switch (code) {
    case ZERO_OK: base = "ok"; break;
    case ZERO_EINVAL: base = "invalid argument (NULL pointer, negative count or bad flag)"; break;
    case ZERO_EALIGN: base = "device array not aligned to 16 bytes"; break;
    case ZERO_EDTYPE: base = "element type not accepted for this argument"; break;
    case ZERO_ESIZE: base = "element counts differ across the lists"; break;
    case ZERO_EWORKSPACE: base = "workspace missing or smaller than zero_workspace_bytes()"; break;
    case ZERO_ECAPACITY: base = "output array too small"; break;
    case ZERO_ECUDA: base = "CUDA runtime error"; break;
    case ZERO_ELAYOUT: base = "bad layout parameters (nd < 1, align not a power of two, or too large)"; break;
    case ZERO_ECAPTURE:
        base = "this call copies a host table, which a stream capture cannot hold; issue it outside capture";
        break;
    default: base = "unknown error code"; break;
    }
    if (code == ZERO_ECUDA && zpml::g_err[0])
        std::snprintf(buf, sizeof buf, "%s: %s", base, zpml::g_err);
    else
        std::snprintf(buf, sizeof buf, "%s", base);
    return buf;
}

extern "C" int zero_partition_layout(const int64_t *numel, int64_t n_tensors, int32_t nd,
                                     int64_t align, int64_t *shard_numel, int64_t *padded_total,
                                     int64_t *tensor_offset, zero_frag_t *frags, int64_t frag_cap,
                                     int64_t *n_frags)
{
    if (n_tensors < 0 || (n_tensors > 0 && !numel) || !shard_numel || !padded_total || !n_frags ||
        frag_cap < 0 || (frag_cap > 0 && !frags))
        return ZERO_EINVAL;
    if (nd < 1 || align < 1 || (align & (align - 1)) != 0)
        return ZERO_ELAYOUT;
    const int64_t kLimit = (int64_t)1 << 62;
    int64_t total = 0;
    for (int64_t i = 0; i < n_tensors; ++i) {
        if (numel[i] < 0)
            return ZERO_EINVAL;
        if (numel[i] > kLimit - total)
            return ZERO_ELAYOUT;
        total += numel[i];
    }
    if (align > kLimit / nd)
        return ZERO_ELAYOUT;
    const int64_t unit = (int64_t)nd * align;
    const int64_t units = total / unit + (total % unit != 0);
    if (units > kLimit / unit)
        return ZERO_ELAYOUT;
    const int64_t shard = units * align;

    // Walk the flat buffer once: each tensor is cut at every shard boundary
    // that falls inside it.
    int64_t count = 0, off = 0;
    for (int64_t t = 0; t < n_tensors; ++t) {
        if (tensor_offset)
            tensor_offset[t] = off;
        int64_t pos = off;
        const int64_t end = off + numel[t];
        while (pos < end) {
            const int64_t r = pos / shard;
            const int64_t rank_end = (r + 1) * shard;
            const int64_t stop = end < rank_end ? end : rank_end;
            if (count < frag_cap) {
                zero_frag_t &f = frags[count];
                f.tensor = t;
                f.tensor_offset = pos - off;
                f.rank = r;
                f.shard_offset = pos - r * shard;
                f.length = stop - pos;
            }
            ++count;
            pos = stop;
        }
        off = end;
    }
    *shard_numel = shard;
    *padded_total = shard * nd;
    *n_frags = count;
    return count > frag_cap ? ZERO_ECAPACITY : ZERO_OK;
}

extern "C" int zero_state_init(zero_state_t *s, double initial_loss_scale)
{
    if (!s || !(initial_loss_scale >= 1.0) || !std::isfinite(initial_loss_scale))
        return ZERO_EINVAL;
    int e = 0;
    if (std::frexp(initial_loss_scale, &e) != 0.5)  // must be a power of two
        return ZERO_EINVAL;
    std::memset(s, 0, sizeof *s);
    s->loss_scale = initial_loss_scale;
    s->last_clip = 1.0f;
    return ZERO_OK;
}

extern "C" size_t zero_workspace_bytes(int64_t max_tensors, int64_t max_total_numel)
{
    if (max_tensors < 1)
        max_tensors = 1;
    if (max_total_numel < 0)
        max_total_numel = 0;
    return zpml::kWsTable + zpml::table_bytes(max_tensors, max_total_numel);
}

// Stage-3 gather plan.  Same source, same section: stage 3 partitions the
// parameters too, so each layer's parameters are gathered from the ranks'
// shards before the layer runs.  A layer's tensors are consecutive in the
// flat buffer, so the layer is one flat range and meets each rank's shard in
// at most one contiguous piece.
extern "C" int zero_gather_plan(const int64_t *numel, int64_t n_tensors, const int64_t *layer_first,
                                int64_t n_layers, int32_t nd, int64_t align, int64_t *layer_flat,
                                zero_gather_piece_t *pieces, int64_t cap, int64_t *n_pieces,
                                int64_t *max_layer_numel)
{
    if (n_layers < 0 || (n_layers > 0 && !layer_first) || !n_pieces || cap < 0 || (cap > 0 && !pieces) ||
        n_tensors < 0)
        return ZERO_EINVAL;
    for (int64_t L = 0; L <= n_layers && n_layers > 0; ++L) {
        const int64_t a = layer_first[L];
        if (a < 0 || a > n_tensors || (L > 0 && a < layer_first[L - 1]))
            return ZERO_ELAYOUT;
    }
    std::vector<int64_t> offs((size_t)n_tensors + 1);
    int64_t shard = 0, padded = 0, n_frags = 0;
    const int rc = zero_partition_layout(numel, n_tensors, nd, align, &shard, &padded, offs.data(), nullptr, 0,
                                         &n_frags);
    if (rc != ZERO_OK && rc != ZERO_ECAPACITY)
        return rc;
    int64_t total = 0;
    for (int64_t i = 0; i < n_tensors; ++i)
        total += numel[i];
    offs[(size_t)n_tensors] = total;

    int64_t count = 0, biggest = 0;
    for (int64_t L = 0; L < n_layers; ++L) {
        const int64_t begin = offs[(size_t)layer_first[L]], end = offs[(size_t)layer_first[L + 1]];
        if (layer_flat)
            layer_flat[L] = begin;
        if (end - begin > biggest)
            biggest = end - begin;
        if (begin == end)
            continue;
        for (int64_t r = begin / shard; r * shard < end; ++r) {
            const int64_t lo = begin > r * shard ? begin : r * shard;
            const int64_t hi = end < (r + 1) * shard ? end : (r + 1) * shard;
            if (count < cap) {
                zero_gather_piece_t &p = pieces[count];
                p.layer = L;
                p.rank = r;
                p.shard_offset = lo - r * shard;
                p.length = hi - lo;
                p.layer_offset = lo - begin;
            }
            ++count;
        }
    }
    if (layer_flat && n_layers > 0)
        layer_flat[n_layers] = offs[(size_t)layer_first[n_layers]];
    if (max_layer_numel)
        *max_layer_numel = biggest;
    *n_pieces = count;
    return count > cap ? ZERO_ECAPACITY : ZERO_OK;
}
