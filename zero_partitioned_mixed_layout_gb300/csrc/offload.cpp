// Host side of a ZeRO-Offload step: the optimizer state (fp32 master,
// momentum, variance) lives in host memory and the host cores update it,
// while the GPU keeps the fp16 parameters and computes the gradient norm.
//
// Source: DeepSpeed release news (lxsoso.com/blog/19320.html): ZeRO-Offload
// extends ZeRO-2 to use CPU memory as well as GPU memory, so that one GPU
// trains a model about ten times larger (13B parameters on one V100);
// "微软|ZeRO-Infinity和DeepSpeed" (hub.baai.ac.cn): the offload engine moves
// partitioned model states to CPU memory.  On GB300 the host is a Grace CPU
// joined to the GPU by NVLink-C2C.
//
// The element update is the library's: the same binary32 expression,
// evaluated operation by operation (this file is built with
// -ffp-contract=off and without fast-math, so no multiply-add is fused), and
// the same step decision with the same binary64 scalars.  Work is split over
// a persistent pool of host threads in chunks of 64 Ki elements.
#include <atomic>
#include <cmath>
#include <condition_variable>
#include <cstring>
#include <functional>
#include <mutex>
#include <thread>
#include <vector>

#include "zero_pml_internal.h"

namespace zpml {
namespace {

constexpr int64_t kHostChunk = 1 << 16;
constexpr int kMaxHostThreads = 256;

// A fixed set of worker threads that run one job at a time; the calling
// thread takes part, so a job on T threads wakes T - 1 workers.
class Pool {
public:
    static Pool &get()
    {
        static Pool pool;
        return pool;
    }

    // Runs fn(i) for every i in [0, n_items) on up to n_threads threads.
    void run(int64_t n_items, int n_threads, const std::function<void(int64_t)> &fn)
    {
        std::lock_guard<std::mutex> one_job(call_mu_);
        if (n_threads < 1)
            n_threads = 1;
        if (n_threads > kMaxHostThreads)
            n_threads = kMaxHostThreads;
        if ((int64_t)n_threads > n_items)
            n_threads = (int)(n_items > 0 ? n_items : 1);
        const int helpers = n_threads - 1;
        {
            std::lock_guard<std::mutex> lk(mu_);
            while ((int)workers_.size() < helpers) {
                const int idx = (int)workers_.size();
                workers_.emplace_back([this, idx] { loop(idx); });
            }
            job_ = &fn;
            n_items_ = n_items;
            next_.store(0);
            want_ = helpers;
            active_ = helpers;
            ++gen_;
        }
        cv_.notify_all();
        work();
        std::unique_lock<std::mutex> lk(mu_);
        done_cv_.wait(lk, [this] { return active_ == 0; });
        job_ = nullptr;
    }

    ~Pool()
    {
        {
            std::lock_guard<std::mutex> lk(mu_);
            stop_ = true;
        }
        cv_.notify_all();
        for (auto &t : workers_)
            t.join();
    }

private:
    void work()
    {
        for (int64_t i = next_.fetch_add(1); i < n_items_; i = next_.fetch_add(1))
            (*job_)(i);
    }

    void loop(int idx)
    {
        uint64_t seen = 0;
        std::unique_lock<std::mutex> lk(mu_);
        for (;;) {
            cv_.wait(lk, [&] { return stop_ || (gen_ != seen && idx < want_); });
            if (stop_)
                return;
            seen = gen_;
            lk.unlock();
            work();
            lk.lock();
            if (--active_ == 0)
                done_cv_.notify_one();
        }
    }

    std::mutex call_mu_, mu_;
    std::condition_variable cv_, done_cv_;
    std::vector<std::thread> workers_;
    const std::function<void(int64_t)> *job_ = nullptr;
    int64_t n_items_ = 0;
    std::atomic<int64_t> next_{0};
    int want_ = 0, active_ = 0;
    uint64_t gen_ = 0;
    bool stop_ = false;
};

// binary16 -> binary32, exact, in integer and binary32 operations that the
// compiler vectorises (a _Float16 conversion is not vectorised for the
// generic Arm target): the exponent and mantissa move to the binary32
// positions and one exact multiplication by 2^112 rebiases the exponent (a
// subnormal half becomes a subnormal single before the multiplication and a
// normal one after it); an all-ones exponent (inf, NaN) maps to all ones.
// NaN payloads are kept as they are (a skipped step never reads them).
inline float from_f16(uint16_t b)
{
    const uint32_t em = (uint32_t)(b & 0x7FFFu) << 13;
    float f;
    std::memcpy(&f, &em, sizeof f);
    f = f * 0x1p112f;
    uint32_t r;
    std::memcpy(&r, &f, sizeof r);
    const uint32_t special = 0u - (uint32_t)((b & 0x7C00u) == 0x7C00u);  // all ones for inf / NaN
    r = (r & ~special) | ((em | 0x7F800000u) & special);
    r |= (uint32_t)(b & 0x8000u) << 16;
    float out;
    std::memcpy(&out, &r, sizeof out);
    return out;
}

inline uint16_t to_f16(float x)
{
    const _Float16 h = (_Float16)x;  // IEEE conversion, round to nearest even
    uint16_t b;
    std::memcpy(&b, &h, sizeof b);
    return b;
}

inline float from_bf16(uint16_t b)
{
    const uint32_t u = (uint32_t)b << 16;
    float f;
    std::memcpy(&f, &u, sizeof f);
    return f;
}

// binary32 -> bfloat16, round to nearest even (NaN stays NaN, quiet).
// Written without a branch so that the update loop vectorises.
inline uint16_t to_bf16(float x)
{
    uint32_t u;
    std::memcpy(&u, &x, sizeof u);
    const uint32_t rounded = (u + 0x7FFFu + ((u >> 16) & 1u)) >> 16;
    const uint32_t quiet = (u >> 16) | 0x40u;
    return (uint16_t)(x != x ? quiet : rounded);
}

// The element update, binary32, each operation rounded on its own.
inline void update(float graw, float &p, float &m, float &v, const zero_offload_scalars_t &s)
{
    const float g = (graw * s.inv_scale) * s.clip;
    const float m1 = s.beta1 * m + s.one_minus_beta1 * g;
    const float v1 = s.beta2 * v + s.one_minus_beta2 * (g * g);
    const float d = std::sqrt(v1) * s.inv_sqrt_bc2 + s.eps;
    const float u = m1 / d;
    p = p - (s.step_size * u + s.lr_wd * p);
    m = m1;
    v = v1;
}

enum { kNoLowP = -1 };

template <int GT>
inline float load_g(const void *__restrict__ g, int64_t i)
{
    if (GT == ZERO_F16)
        return from_f16(static_cast<const uint16_t *>(g)[i]);
    if (GT == ZERO_BF16)
        return from_bf16(static_cast<const uint16_t *>(g)[i]);
    return static_cast<const float *>(g)[i];
}

// One chunk [b, e) for one pair of element types: a plain counted loop over
// restrict pointers that the compiler vectorises.
template <int GT, int PT>
void apply_span(const void *__restrict__ g, float *__restrict__ p, float *__restrict__ m, float *__restrict__ v,
                uint16_t *__restrict__ lp, int64_t b, int64_t e, const zero_offload_scalars_t &s)
{
    for (int64_t i = b; i < e; ++i) {
        float pi = p[i], mi = m[i], vi = v[i];
        update(load_g<GT>(g, i), pi, mi, vi, s);
        p[i] = pi;
        m[i] = mi;
        v[i] = vi;
        if (PT == ZERO_F16)
            lp[i] = to_f16(pi);
        else if (PT == ZERO_BF16)
            lp[i] = to_bf16(pi);
    }
}

template <int GT>
void apply_lp(int32_t pdtype, const void *g, float *p, float *m, float *v, uint16_t *lp, int64_t b, int64_t e,
              const zero_offload_scalars_t &s)
{
    if (!lp)
        apply_span<GT, kNoLowP>(g, p, m, v, lp, b, e, s);
    else if (pdtype == ZERO_BF16)
        apply_span<GT, ZERO_BF16>(g, p, m, v, lp, b, e, s);
    else
        apply_span<GT, ZERO_F16>(g, p, m, v, lp, b, e, s);
}

}  // namespace
}  // namespace zpml

using namespace zpml;

extern "C" int zero_offload_decide(zero_state_t *st, const zero_hparams_t *hp, zero_offload_scalars_t *out)
{
    if (!st || !hp || !out)
        return ZERO_EINVAL;
    if (!(hp->lr >= 0.0) || !(hp->beta1 >= 0.0 && hp->beta1 < 1.0) || !(hp->beta2 >= 0.0 && hp->beta2 < 1.0) ||
        !(hp->eps >= 0.0) || !(hp->weight_decay >= 0.0) || !(hp->min_scale >= 1.0) || hp->scale_window < 1 ||
        hp->max_norm != hp->max_norm || !(st->loss_scale >= 1.0))
        return ZERO_EINVAL;
    int e = 0;
    if (!std::isfinite(hp->min_scale) || std::frexp(hp->min_scale, &e) != 0.5)  // a power of two
        return ZERO_EINVAL;
    zero_offload_scalars_t o;
    std::memset(&o, 0, sizeof o);
    o.inv_scale = (float)(1.0 / st->loss_scale);
    o.clip = 1.0f;
    const double norm = std::sqrt(st->sumsq);
    if (st->found_inf != 0.0) {
        o.skip = 1;
        const double half = st->loss_scale * 0.5;
        st->loss_scale = half < hp->min_scale ? hp->min_scale : half;
        st->good_steps = 0;
        st->skipped += 1;
    } else {
        st->step += 1;
        st->good_steps += 1;
        if (st->good_steps >= hp->scale_window) {
            st->loss_scale *= 2.0;
            st->good_steps = 0;
        }
        double clip = 1.0;
        if (hp->max_norm > 0.0) {
            const double c = hp->max_norm / (norm + 1e-6);
            if (c < 1.0)
                clip = c;
        }
        const double t = (double)st->step;
        const double bc1 = 1.0 - std::pow(hp->beta1, t);
        const double bc2 = 1.0 - std::pow(hp->beta2, t);
        o.clip = (float)clip;
        o.beta1 = (float)hp->beta1;
        o.one_minus_beta1 = (float)(1.0 - hp->beta1);
        o.beta2 = (float)hp->beta2;
        o.one_minus_beta2 = (float)(1.0 - hp->beta2);
        o.eps = (float)hp->eps;
        o.step_size = (float)(hp->lr / bc1);
        o.inv_sqrt_bc2 = (float)(1.0 / std::sqrt(bc2));
        o.lr_wd = (float)(hp->lr * hp->weight_decay);
    }
    st->last_norm = norm;
    st->last_clip = o.clip;
    st->last_skipped = o.skip;
    st->sumsq = 0.0;
    st->found_inf = 0.0;
    *out = o;
    return ZERO_OK;
}

extern "C" int zero_offload_apply(const void *grad, int32_t gdtype, float *master, float *m, float *v,
                                  void *p_lp, int32_t pdtype, int64_t n, const zero_offload_scalars_t *sc,
                                  int32_t n_threads)
{
    if (n < 0 || !sc || n_threads < 1)
        return ZERO_EINVAL;
    if (gdtype != ZERO_F16 && gdtype != ZERO_BF16 && gdtype != ZERO_F32)
        return ZERO_EDTYPE;
    if (p_lp && pdtype != ZERO_F16 && pdtype != ZERO_BF16)
        return ZERO_EDTYPE;
    if (n == 0 || sc->skip)
        return ZERO_OK;
    if (!grad || !master || !m || !v)
        return ZERO_EINVAL;
    const zero_offload_scalars_t s = *sc;
    const int64_t chunks = (n + kHostChunk - 1) / kHostChunk;
    uint16_t *lp = static_cast<uint16_t *>(p_lp);
    std::function<void(int64_t)> job = [&](int64_t c) {
        const int64_t b = c * kHostChunk, e = b + kHostChunk < n ? b + kHostChunk : n;
        if (gdtype == ZERO_F16)
            apply_lp<ZERO_F16>(pdtype, grad, master, m, v, lp, b, e, s);
        else if (gdtype == ZERO_BF16)
            apply_lp<ZERO_BF16>(pdtype, grad, master, m, v, lp, b, e, s);
        else
            apply_lp<ZERO_F32>(pdtype, grad, master, m, v, lp, b, e, s);
    };
    Pool::get().run(chunks, n_threads, job);
    return ZERO_OK;
}

extern "C" int zero_offload_copy(void *dst, const void *src, size_t bytes, int32_t n_threads)
{
    if ((bytes > 0 && (!dst || !src)) || n_threads < 1)
        return ZERO_EINVAL;
    const size_t piece = (size_t)1 << 20;
    const int64_t pieces = (int64_t)((bytes + piece - 1) / piece);
    std::function<void(int64_t)> job = [&](int64_t k) {
        const size_t b = (size_t)k * piece, e = b + piece < bytes ? b + piece : bytes;
        std::memcpy(static_cast<char *>(dst) + b, static_cast<const char *>(src) + b, e - b);
    };
    Pool::get().run(pieces, n_threads, job);
    return ZERO_OK;
}
