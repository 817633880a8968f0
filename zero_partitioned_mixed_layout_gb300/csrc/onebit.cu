// 1-bit Adam's compression stage on one rank: the worker side (local
// momentum, error feedback, compression to signs and one scale), the server
// side for the rank's chunk (the workers' mean, error feedback,
// recompression) and the update with the frozen variance.
//
// Source: DeepSpeed release news (lxsoso.com/blog/19320.html) names 1-bit
// Adam: up to 5x less communication than Adam with Adam's convergence.  The
// page gives no algorithm; the steps follow the outline of the published
// method (Tang et al. 2021): warm-up with plain Adam, then a frozen variance
// and a momentum all-reduce compressed to one bit per element with error
// feedback on the workers and on the servers.
//
// Every pass streams HBM.  A compression needs the L2 norm of its whole
// input before any sign can be turned into an error, and a second pass over
// the input would cost 8 bytes per element more.  So the error is kept in
// deferred form: the state array holds the compression's input x itself and
// the scale array its scale s, and the error x - s*sign(x) is formed (one
// binary32 subtraction, the same as forming it at once) when the next step
// reads x.  One pass then reads the previous x, forms the new input and
// writes it, its signs (packed 32 to a word with two warp shuffles) and its
// squared norm (binary32 squares summed per 8 elements and range-checked,
// one binary64 add per 32 elements, fixed-order block partials, the last
// block finishing the sum and writing the new scale).  Bytes per element with an fp16 gradient:
// worker 2 + 1/8 + 8 + 1/8 with the momentum as the servers' signs (2 + 4 +
// 8 + 1/8 with a dense one); server Nd/8 + 8 + 1/8 per chunk element;
// update 1/8 + 12 + 2 (+ 4 with a dense momentum written).
#include <vector>

#include "common.cuh"

namespace zpml {
namespace {

// 8 binary32 values at p with streaming (evict-first) hints: one 32-byte
// access when p is on a 32-byte boundary (W32), else two 16-byte ones.  The
// 32-byte form matters for the fused compression passes: with two 16-byte
// accesses a lane's instruction covers half of each 32-byte sector, and the
// worker pass measured 2.2-5.8 TB/s depending on how the compiler placed
// the two halves, against 6.7 TB/s with one 32-byte access.
template <bool W32>
__device__ __forceinline__ void ld8(const float *p, float *f)
{
    if constexpr (W32) {
        asm("ld.global.cs.v8.f32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
            : "=f"(f[0]), "=f"(f[1]), "=f"(f[2]), "=f"(f[3]), "=f"(f[4]), "=f"(f[5]), "=f"(f[6]), "=f"(f[7])
            : "l"(p));
    } else {
        const float4 a = __ldcs(reinterpret_cast<const float4 *>(p));
        const float4 b = __ldcs(reinterpret_cast<const float4 *>(p) + 1);
        f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
        f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
    }
}

template <bool W32>
__device__ __forceinline__ void st8(float *p, const float *f)
{
    if constexpr (W32) {
        asm volatile("st.global.cs.v8.f32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "f"(f[0]), "f"(f[1]),
                     "f"(f[2]), "f"(f[3]), "f"(f[4]), "f"(f[5]), "f"(f[6]), "f"(f[7])
                     : "memory");
    } else {
        __stcs(reinterpret_cast<float4 *>(p), make_float4(f[0], f[1], f[2], f[3]));
        __stcs(reinterpret_cast<float4 *>(p) + 1, make_float4(f[4], f[5], f[6], f[7]));
    }
}

bool aligned32(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 31u) == 0; }

// End of a squared-norm pass: publish this block's partial; the block that
// takes the last ticket sums the partials in block order and writes the
// compressor's scale sqrt(sum / len), rounded once to binary32 (not on a
// skipped step, whose blocks still pass here to keep the ticket in step).
__device__ void scale_finish(double tot, double2 *partials, WsHeader *hdr, int64_t len, float *scale, bool skip)
{
    __shared__ bool s_last;
    uint32_t none = 0;
    block_reduce(tot, none);
    if (threadIdx.x == 0) {
        partials[blockIdx.x] = make_double2(tot, 0.0);
        __threadfence();
        s_last = atomicAdd(&hdr->ticket, 1u) == gridDim.x - 1;
    }
    __syncthreads();
    if (!s_last)
        return;
    __threadfence();
    double t = 0.0;
    for (int j = threadIdx.x; j < (int)gridDim.x; j += kThreads)
        t += __ldcg(partials + j).x;
    block_reduce(t, none);
    if (threadIdx.x == 0) {
        if (!skip)
            *scale = (float)sqrt(t / (double)len);
        hdr->ticket = 0u;
    }
}

// Squares of one 8-element group into a binary32 lane sum; every 4 groups
// (32 elements) the lane sum goes into the binary64 total.  The compressed
// values are binary32 of any size, so each group's binary32 sum is
// range-checked and an out-of-range group's squares go to the binary64
// total directly (add_squares_checked).
struct SquareSum {
    double tot = 0.0;
    float part = 0.0f;
    int groups = 0;
    __device__ __forceinline__ void add(const float *x)
    {
        add_squares_checked(x, nonzero8(x), part, tot);
        if (++groups == 4) {
            tot += (double)part;
            part = 0.0f;
            groups = 0;
        }
    }
    __device__ __forceinline__ double total() const { return tot + (double)part; }
    // The first `count` of 4 vectors (32 elements) still in registers: their
    // squares by FMA in 8 binary32 lanes and one range check of the lanes'
    // sum (finite, and at least 2^-90 unless every value is zero); an
    // out-of-range group is summed again in binary64.
    __device__ __forceinline__ void add4(const float (*y)[8], int count)
    {
        float lanes[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        uint32_t nz = 0;
#pragma unroll
        for (int v = 0; v < 4; ++v) {
            if (v < count) {
                nz |= nonzero8(y[v]);
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    lanes[k] = __fmaf_rn(y[v][k], y[v][k], lanes[k]);
            }
        }
        const float s = tree8(lanes);
        if (s < __int_as_float(0x7F800000) && (s >= 0x1p-90f || nz == 0u)) {
            tot += (double)s;
        } else {
#pragma unroll
            for (int v = 0; v < 4; ++v)
                if (v < count)
                    tot += squares_wide(y[v]);
        }
    }
};

// The error a compression left, from its input x and scale sc: x - sc where
// x is not negative (sign +1, also for -0), x + sc where it is.
__device__ __forceinline__ float deferred_error(float x, float sc)
{
    return __fsub_rn(x, !(x < 0.0f) ? sc : -sc);
}

// Sign bits of one 8-element group: bit k for element k, 1 where the value
// is not negative (-0 counts as +).
__device__ __forceinline__ uint32_t sign_byte(const float *x)
{
    uint32_t byte = 0;
#pragma unroll
    for (int k = 0; k < 8; ++k)
        byte |= (uint32_t)!(x[k] < 0.0f) << k;
    return byte;
}

// The word of 32 signs that four consecutive lanes' bytes make (lane & 3 =
// the byte's place in the word); warp code, every lane calls it.
__device__ __forceinline__ uint32_t sign_word(uint32_t byte)
{
    uint32_t w = byte << (8 * (threadIdx.x & 3));
    w |= __shfl_xor_sync(0xffffffffu, w, 1);
    w |= __shfl_xor_sync(0xffffffffu, w, 2);
    return w;
}

// The skip flag of these kernels comes from device memory.  They do not
// return early on it: a data-dependent exit ahead of the block barriers of
// the reduction cost a third of the streaming rate of the loop on GB300 (the
// same loop with the flag as a kernel argument, or folded into the loop
// bound as here, runs at the copy rate).  A skipped step runs no
// iterations and writes nothing.

// The synchronised momentum of one 8-element group: dense (fp32 array) or
// compressed (the previous step's server signs and per-chunk scales, the
// form the update produces: every element is +-scale of its chunk).
struct Momentum {
    const float *dense;    // or NULL
    const uint32_t *bits;  // compressed form
    const float *scales;
    int64_t chunk;         // S
};

// ci: the chunk of group i, (8i) / S, computed by the caller ahead of its
// loads (so that the division does not sit between them).
template <bool kCompressed, bool W32>
__device__ __forceinline__ void load_momentum(const Momentum &mm, int64_t i, int64_t ci, float *f)
{
    if constexpr (kCompressed) {
        const uint32_t byte = (__ldg(mm.bits + (i >> 2)) >> (8 * (i & 3))) & 0xFFu;
        const float sc = __ldg(mm.scales + ci);
#pragma unroll
        for (int k = 0; k < 8; ++k)
            f[k] = ((byte >> k) & 1u) ? sc : -sc;
    } else {
        ld8<W32>(mm.dense + 8 * i, f);
    }
}

// Worker: x = b1*m + (1-b1)*g + e (g unscaled, clipped), e the error the
// previous compression left in deferred form (its input xs over which x is
// stored, and its scale, read here before this compression's scale replaces
// it); the signs of x and its squared norm into the new scale.  A warp's
// lanes hold 32 consecutive 8-element groups, so that four lanes make one
// word of signs.
template <int GT, bool kCompressed, bool W32>
__global__ void __launch_bounds__(kThreads) k_onebit_worker(const void *g, Momentum mm, float *xs, int64_t n,
                                                            const StepScalars *scp, double2 *partials,
                                                            WsHeader *hdr, float *scale, uint32_t *bits)
{
    pdl_wait();
    const StepScalars s = load_scalars(scp);
    // every block reads the old scale before its ticket; the new one is
    // written by the last block, after every ticket
    const float prev = *scale;
    constexpr int W = Elem<GT>::kWords;
    const uint4 *gv = static_cast<const uint4 *>(g);
    SquareSum acc;
    const int64_t nv = s.skip ? 0 : n >> 3;
    const int64_t stride = (int64_t)gridDim.x * kThreads;
    // the loop runs warp by warp (i0 is the warp's first group), so that the
    // shuffles of the sign words see every lane
    for (int64_t i0 = (int64_t)blockIdx.x * kThreads + (threadIdx.x & ~31); i0 < nv; i0 += stride) {
        const int64_t i = i0 + (threadIdx.x & 31);
        const int64_t ci = kCompressed ? (8 * i) / mm.chunk : 0;
        uint32_t byte = 0;
        if (i < nv) {
            uint4 w[W];
#pragma unroll
            for (int q = 0; q < W; ++q)
                w[q] = __ldcs(gv + i * W + q);
            float gf[8], mf[8], x[8];
            Elem<GT>::to_float(w, gf);
            load_momentum<kCompressed, W32>(mm, i, ci, mf);
            ld8<W32>(xs + 8 * i, x);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const float gk = __fmul_rn(__fmul_rn(gf[k], s.inv_scale), s.clip);
                const float mk = __fadd_rn(__fmul_rn(s.b1, mf[k]), __fmul_rn(s.omb1, gk));
                x[k] = __fadd_rn(mk, deferred_error(x[k], prev));
            }
            st8<W32>(xs + 8 * i, x);
            acc.add(x);
            byte = sign_byte(x);
        }
        const uint32_t word = sign_word(byte);
        if ((threadIdx.x & 3) == 0 && i < nv)
            bits[i >> 2] = word;
    }
    scale_finish(acc.total(), partials, hdr, n, scale, s.skip != 0);
}

// Server over the chunk: y = (sum over workers in rank order of +-scale_k)
// / Nd + f, f the error the previous compression left in deferred form (its
// input ys over which y is stored, and its scale); the signs of y and its
// squared norm into the new scale.
//
// Per element the sum is Nd dependent binary32 additions, which would make
// the pass bound by instruction issue rather than by memory.  But an element
// enters the sum only through its Nd signs, and the scales are the same for
// the whole chunk: so each block first tabulates, in shared memory, the
// rank-order sum for every sign pattern of the first P = min(Nd, 14) workers
// (2^P binary32 values, built one worker at a time with the very additions
// an element would make), and an element then looks its first P signs up
// and adds the remaining workers' terms in rank order.  Same additions,
// same order, same bits.
//
// Data movement: a warp takes 1024 elements (32 words of signs, 128 vectors
// of 8) at a time.  Lane l loads the 16 workers' sign words of word l
// (coalesced: a warp's loads of one worker are one 128-byte line) and turns
// them around with one 16x32 bit-matrix transpose in registers into each of
// the word's 32 elements' 16-bit sign pattern; the patterns go through 2 KB
// of shared memory per warp to the lanes that hold those elements' values,
// which are read and written coalesced (lane l holds vectors l + 32v).  The
// staging is swizzled so that both sides are free of bank conflicts.
// Workers past 16 go the same way, 16 at a time.  Bytes per chunk element:
// Nd/8 + 4 + 4 + 1/8.
constexpr int kTableBits = 14;
// Workers per server call: their pointers and scales (12 bytes each) and
// the 64 KiB table fit in shared memory.
constexpr int kMaxServerWorkers = 4096;
// Workers whose sign pointers travel as a launch argument (no table copy,
// so that the call can be captured into a graph).
constexpr int kArgWorkers = 256;
struct WorkerPtrs {
    const uint32_t *p[kArgWorkers];
};

// The signs of 16 workers for the 32 elements of one word, turned around:
// on entry W[k] holds worker k's word (bit e for element e); on return the
// low half of W[i] holds element i's signs and the high half element
// 16 + i's, bit k for worker k.  A 16x16 bit-matrix transpose of each half
// at once, by the recursive block swap (Hacker's Delight, section 7-3):
// four stages that exchange the off-diagonal s x s blocks (s = 8, 4, 2, 1)
// of every 2s x 2s block, five integer operations per row pair.
template <int S, uint32_t M>
__device__ __forceinline__ void transpose16_stage(uint32_t *W)
{
#pragma unroll
    for (int r = 0; r < 16; ++r) {
        if ((r & S) == 0) {
            const uint32_t t = ((W[r] >> S) ^ W[r + S]) & M;
            W[r + S] ^= t;
            W[r] ^= t << S;
        }
    }
}

// The stages with their shifts and masks as constants, so that every row
// index is fixed at compile time and the rows stay in registers.
__device__ __forceinline__ void transpose16(uint32_t *W)
{
    transpose16_stage<8, 0x00FF00FFu>(W);
    transpose16_stage<4, 0x0F0F0F0Fu>(W);
    transpose16_stage<2, 0x33333333u>(W);
    transpose16_stage<1, 0x55555555u>(W);
}

// +scale where the sign bit (at bit 31 of t) is set, -scale where it is
// clear: the scale's bits with the sign bit flipped.
__device__ __forceinline__ float signed_scale(uint32_t scale_bits, uint32_t t)
{
    return __uint_as_float(scale_bits ^ (~t & 0x80000000u));
}

// The dynamic shared memory of the server: the table, the worker pointers
// and the scales.
// Per warp: 32 lanes x 32 elements x 2 bytes of staged sign patterns.
constexpr size_t kStageBytesPerWarp = 2048;

__host__ __device__ constexpr size_t server_smem_bytes(int nd)
{
    return kStageBytesPerWarp * kWarps + sizeof(float) * ((size_t)1 << (nd < kTableBits ? nd : kTableBits)) +
           (sizeof(void *) + sizeof(float)) * (size_t)nd;
}

// The 16-byte slot of staging chunk c (chunk 4w + q: the sign patterns of
// elements 8q .. 8q+7 of the warp's word w): the low two bits of the 16-byte
// bank group are XORed with bits 3-4 of c, so that the writes (lane w: chunks
// 4w + q) and the reads (lane l: chunk l + 32v) each spread over all eight
// bank groups.
__device__ __forceinline__ int stage_slot(int c) { return c ^ ((c >> 3) & 3); }

// Lane side of the staging: the 16 sign words W (after transpose16) of this
// lane's word w, packed two patterns to a 32-bit word in element order, into
// the warp's staging area.
__device__ __forceinline__ void stage_patterns(const uint32_t *W, uint4 *stage, int lane)
{
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        // elements 8q .. 8q+7: low halves of rows 0-7 / 8-15 for q = 0 / 1,
        // high halves for q = 2 / 3
        const int r0 = (q & 1) * 8;
        const uint32_t sel = q < 2 ? 0x5410u : 0x7632u;
        uint4 c;
        c.x = __byte_perm(W[r0 + 0], W[r0 + 1], sel);
        c.y = __byte_perm(W[r0 + 2], W[r0 + 3], sel);
        c.z = __byte_perm(W[r0 + 4], W[r0 + 5], sel);
        c.w = __byte_perm(W[r0 + 6], W[r0 + 7], sel);
        stage[stage_slot(4 * lane + q)] = c;
    }
}

// The rank-order sums over workers 0-15 of one vector's 8 elements from
// their staged sign patterns (pc: element j's pattern in half j & 1 of word
// j >> 1): the table entry for workers 0..P-1, then workers 14 and 15.
__device__ __forceinline__ void first16_sums(uint4 pc, const float *T, uint32_t pmask, int P, int upto16,
                                             uint32_t sb14, uint32_t sb15, float *a)
{
    const uint32_t pw[4] = {pc.x, pc.y, pc.z, pc.w};
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        // element j's pattern in bits 0-15 of t (16-31 of pw)
        const uint32_t t = (j & 1) ? pw[j >> 1] >> 16 : pw[j >> 1];
        float x = T[t & pmask];
        if (P == 14 && upto16 > 14)
            x = __fadd_rn(x, signed_scale(sb14, t << 17));
        if (P == 14 && upto16 > 15)
            x = __fadd_rn(x, signed_scale(sb15, t << 16));
        a[j] = x;
    }
}

// One vector (elements 8i .. 8i+7) of the chunk: the mean of its sums plus
// the error the previous compression left, stored (its squares are summed
// with the lane's other vectors at the end of the chunk); its signs, one
// byte, four lanes' bytes making one word.  Warp code (the word's shuffles):
// every lane calls it, i >= nv writes nothing.
template <bool kPow2, bool W32>
__device__ __forceinline__ void finish_vector(const float *a, float *y, int64_t i, int64_t nv, float inv_nd,
                                              float count, float prev, float *ys, uint32_t *bits, int lane)
{
    uint32_t byte = 0;
    if (i < nv) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            // a power-of-two count: the product by its reciprocal is the
            // correctly rounded quotient itself
            const float mean = kPow2 ? __fmul_rn(a[j], inv_nd) : __fdiv_rn(a[j], count);
            y[j] = __fadd_rn(mean, deferred_error(y[j], prev));
        }
        st8<W32>(ys + 8 * i, y);
        byte = sign_byte(y);
    }
    // lanes 4j..4j+3 hold consecutive vectors: one word
    const uint32_t word = sign_word(byte);
    if ((lane & 3) == 0 && i < nv)
        bits[i >> 2] = word;
}

// kWide: more than 16 workers; at most 16, each vector's sums meet their
// values as soon as they are formed (a kernel of its own, with fewer live
// registers).
template <bool kPow2, bool W32, bool kWide>
__device__ __forceinline__ void server_body(const uint32_t *const *wbits, const float *wscales, int nd, float inv_nd,
                                            float *ys, int64_t S, const StepScalars *scp, double2 *partials,
                                            WsHeader *hdr, float *scale, uint32_t *bits)
{
    extern __shared__ __align__(16) unsigned char s_raw[];
    const int P = nd < kTableBits ? nd : kTableBits;
    // dynamic shared memory, in server_smem_bytes' order: the warps' staging
    // areas, the table, the worker pointers, the scales
    uint4 *stage = reinterpret_cast<uint4 *>(s_raw + kStageBytesPerWarp * (threadIdx.x >> 5));
    float *T = reinterpret_cast<float *>(s_raw + kStageBytesPerWarp * kWarps);
    const uint32_t **s_ptr = reinterpret_cast<const uint32_t **>(T + ((size_t)1 << P));
    float *s_scale = reinterpret_cast<float *>(s_ptr + nd);
    pdl_wait();
    // the old scale, read by every block before its ticket
    const float prev = *scale;
    for (int k = threadIdx.x; k < nd; k += kThreads) {
        s_ptr[k] = wbits[k];
        s_scale[k] = wscales[k];
    }
    __syncthreads();
    // T[p] = the rank-order sum over workers k < P of +-scale_k (+ where
    // bit k of p is set), the first term taken as it is
    if (threadIdx.x < 2)
        T[threadIdx.x] = threadIdx.x ? s_scale[0] : -s_scale[0];
    __syncthreads();
    for (int k = 1; k < P; ++k) {
        const int half = 1 << k;
        const float sk = s_scale[k];
        for (int q = threadIdx.x; q < half; q += kThreads) {
            const float t = T[q];
            T[q + half] = __fadd_rn(t, sk);
            T[q] = __fadd_rn(t, -sk);
        }
        __syncthreads();
    }
    const bool skip = load_scalars(scp).skip != 0;
    const int lane = threadIdx.x & 31;
    const uint32_t pmask = (1u << P) - 1u;
    // workers P..15 that the table leaves out (none when Nd <= 14)
    const int upto16 = nd < 16 ? nd : 16;
    const uint32_t sb14 = 14 < upto16 ? __float_as_uint(s_scale[14]) : 0u;
    const uint32_t sb15 = 15 < upto16 ? __float_as_uint(s_scale[15]) : 0u;
    const float count = (float)nd;
    const int64_t nv = skip ? 0 : S >> 3, nw = S >> 5;
    const int64_t chunks = (nv + 127) >> 7;
    SquareSum acc;
    // workers 0-15's sign words of a chunk's word for this lane (zeros past
    // the chunk's end or the worker count)
    auto load_words = [&](int64_t cc, uint32_t *Wd) {
        const int64_t ww = (cc << 5) + lane;
        const bool ok = cc < chunks && ww < nw;
#pragma unroll
        for (int k = 0; k < 16; ++k)
            Wd[k] = k < nd && ok ? __ldg(s_ptr[k] + ww) : 0u;
    };
    const int64_t cstride = (int64_t)gridDim.x * kWarps;
    // up to 16 workers: the next chunk's words are loaded while this chunk is
    // worked on (the wide kernel has no registers to spare for them)
    uint32_t Wn[16];
    if constexpr (!kWide)
        load_words((int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5), Wn);
    for (int64_t c = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5); c < chunks; c += cstride) {
        const int64_t v0 = c << 7, w = (c << 5) + lane;
        const bool wok = w < nw;
        float y[4][8];
#pragma unroll
        for (int v = 0; v < 4; ++v) {
            const int64_t i = v0 + lane + 32 * v;
            if (i < nv)
                ld8<W32>(ys + 8 * i, y[v]);
        }
        // workers 0-15: the table index (bits 0..P-1 of the pattern) and
        // workers 14 and 15 added after it
        {
            uint32_t W[16];
            if constexpr (!kWide) {
#pragma unroll
                for (int k = 0; k < 16; ++k)
                    W[k] = Wn[k];
                load_words(c + cstride, Wn);
            } else {
                load_words(c, W);
            }
            transpose16(W);
            stage_patterns(W, stage, lane);
        }
        __syncwarp();
        if constexpr (!kWide) {
            // each vector's sums meet their values at once: 8 sums live
            // instead of 32
#pragma unroll
            for (int v = 0; v < 4; ++v) {
                const uint4 pc = stage[stage_slot(lane + 32 * v)];
                float a[8];
                first16_sums(pc, T, pmask, P, upto16, sb14, sb15, a);
                finish_vector<kPow2, W32>(a, y[v], v0 + lane + 32 * v, nv, inv_nd, count, prev, ys, bits, lane);
            }
            // the squares of the lane's vectors, still in registers, at once:
            // vector v is v0 + lane + 32v, present while below nv
            const int64_t left = nv - (v0 + lane);
            acc.add4(y, left <= 0 ? 0 : left >= 97 ? 4 : (int)((left + 31) / 32));
            __syncwarp();  // the staging area is reused by the next chunk
            continue;
        }
        float a[4][8];
#pragma unroll
        for (int v = 0; v < 4; ++v)
            first16_sums(stage[stage_slot(lane + 32 * v)], T, pmask, P, upto16, sb14, sb15, a[v]);
        // workers 16 and up, 16 at a time, in rank order
        for (int g = 16; g < nd; g += 16) {
            __syncwarp();  // every lane has read the previous patterns
            {
                uint32_t W[16];
#pragma unroll
                for (int k = 0; k < 16; ++k)
                    W[k] = g + k < nd && wok ? __ldg(s_ptr[g + k] + w) : 0u;
                transpose16(W);
                stage_patterns(W, stage, lane);
            }
            __syncwarp();
            const int nq = nd - g < 16 ? nd - g : 16;
#pragma unroll
            for (int v = 0; v < 4; ++v) {
                const uint4 pc = stage[stage_slot(lane + 32 * v)];
                const uint32_t pw[4] = {pc.x, pc.y, pc.z, pc.w};
#pragma unroll
                for (int q = 0; q < 16; ++q) {
                    if (q < nq) {
                        const uint32_t sb = __float_as_uint(s_scale[g + q]);
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            // worker g + q's sign of element j, moved to bit 31
                            const uint32_t t = (j & 1) ? pw[j >> 1] << (15 - q) : pw[j >> 1] << (31 - q);
                            a[v][j] = __fadd_rn(a[v][j], signed_scale(sb, t));
                        }
                    }
                }
            }
        }
        __syncwarp();  // the staging area is reused by the next chunk
#pragma unroll
        for (int v = 0; v < 4; ++v)
            finish_vector<kPow2, W32>(a[v], y[v], v0 + lane + 32 * v, nv, inv_nd, count, prev, ys, bits, lane);
        const int64_t left = nv - (v0 + lane);
        acc.add4(y, left <= 0 ? 0 : left >= 97 ? 4 : (int)((left + 31) / 32));
    }
    scale_finish(acc.total(), partials, hdr, S, scale, skip);
}

// The worker pointers from a table in the workspace, or as a launch argument.
template <bool kPow2, bool W32>
__global__ void __launch_bounds__(kThreads, 2) k_onebit_server(const uint32_t *const *wbits, const float *wscales,
                                                               int nd, float inv_nd, float *ys, int64_t S,
                                                               const StepScalars *scp, double2 *partials,
                                                               WsHeader *hdr, float *scale, uint32_t *bits)
{
    server_body<kPow2, W32, true>(wbits, wscales, nd, inv_nd, ys, S, scp, partials, hdr, scale, bits);
}

template <bool kPow2, bool W32, bool kWide>
__global__ void __launch_bounds__(kThreads, 2) k_onebit_server_args(const __grid_constant__ WorkerPtrs wp,
                                                                    const float *wscales, int nd, float inv_nd,
                                                                    float *ys, int64_t S, const StepScalars *scp,
                                                                    double2 *partials, WsHeader *hdr, float *scale,
                                                                    uint32_t *bits)
{
    server_body<kPow2, W32, kWide>(wp.p, wscales, nd, inv_nd, ys, S, scp, partials, hdr, scale, bits);
}

// One element of the update with the frozen variance:
//   m = +-scale;  p = p - (step_size * m / (sqrt(v)*isb2 + eps) + lrwd*p)
__device__ __forceinline__ void onebit_elem(float mi, float vi, float &p, const StepScalars &s)
{
    const float d = __fadd_rn(__fmul_rn(__fsqrt_rn(vi), s.isb2), s.eps);
    const float u = __fdiv_rn(mi, d);
    p = __fsub_rn(p, __fadd_rn(__fmul_rn(s.step_size, u), __fmul_rn(s.lrwd, p)));
}

constexpr int kNoLowP = -1;

// The update: one 8-element group per thread (one-shot grid) over the whole
// padded buffer of n = Nd*S elements.  The momentum covers all of it; the
// parameters only the first numel elements (the group that straddles numel
// goes element by element).  m (the dense momentum) is written only when
// given: the next worker can read the momentum in its compressed form.
template <int PT, bool W32>
__global__ void __launch_bounds__(kThreads) k_onebit_update(const uint32_t *bits, const float *scales, int64_t S,
                                                            int64_t n, int64_t numel, float *p, float *m,
                                                            const float *v, void *plp, const StepScalars *scp)
{
    const StepScalars s = load_scalars(scp);
    const int64_t i = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    const int64_t nv = s.skip ? 0 : n >> 3;
    if (i >= nv)
        return;
    const uint32_t byte = (__ldg(bits + (i >> 2)) >> (8 * (i & 3))) & 0xFFu;
    const float sc = __ldg(scales + (8 * i) / S);
    float mf[8];
#pragma unroll
    for (int k = 0; k < 8; ++k)
        mf[k] = ((byte >> k) & 1u) ? sc : -sc;
    if (m)
        st8<W32>(m + 8 * i, mf);
    if (8 * i + 8 <= numel) {
        float vf[8], pf[8];
        ld8<W32>(v + 8 * i, vf);
        ld8<W32>(p + 8 * i, pf);
#pragma unroll
        for (int k = 0; k < 8; ++k)
            onebit_elem(mf[k], vf[k], pf[k], s);
        st8<W32>(p + 8 * i, pf);
        if constexpr (PT != kNoLowP)
            __stcs(reinterpret_cast<uint4 *>(plp) + i, LowP<PT>::pack(pf));
    } else {
        for (int64_t j = 8 * i; j < numel; ++j) {
            float pj = p[j];
            onebit_elem(((byte >> (j - 8 * i)) & 1u) ? sc : -sc, v[j], pj, s);
            p[j] = pj;
            if constexpr (PT != kNoLowP)
                LowP<PT>::store(plp, j, pj);
        }
    }
}

// ------------------------------------------------------------- host side

bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

int check_ws_table(void *ws, size_t ws_bytes, size_t table)
{
    if (!ws)
        return ZERO_EWORKSPACE;
    if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0)
        return ZERO_EALIGN;
    if (ws_bytes < kWsTable + table)
        return ZERO_EWORKSPACE;
    return device_ptr(ws) ? ZERO_OK : ZERO_EINVAL;
}

StepScalars *step_scalars(void *ws)
{
    return reinterpret_cast<StepScalars *>(static_cast<unsigned char *>(ws) + kWsScalars);
}

template <int GT, bool kCompressed, bool W32>
int launch_worker(const void *g, const Momentum &mm, float *xs, int64_t n, uint32_t *bits, float *scale, void *ws,
                  cudaStream_t st)
{
    unsigned char *w = static_cast<unsigned char *>(ws);
    WsHeader *hdr = reinterpret_cast<WsHeader *>(w);
    double2 *partials = reinterpret_cast<double2 *>(w + kWsPartials);
    const StepScalars *sc = step_scalars(ws);
    const int64_t nv = n >> 3;
    auto kern = k_onebit_worker<GT, kCompressed, W32>;
    const int grid = grid_for((const void *)kern, (nv + kThreads - 1) / kThreads, kMaxBlocks, 4);
    launch_k(kern, grid, kThreads, st, true, g, mm, xs, n, sc, partials, hdr, scale, bits);
    return check_launch("zero_onebit_worker");
}

// The worker for the momentum's form and the fp32 arrays' alignment (32
// bytes: one access per 8 elements).
template <int GT>
int launch_worker_m(const void *g, const Momentum &mm, float *xs, int64_t n, uint32_t *bits, float *scale, void *ws,
                    cudaStream_t st)
{
    if (mm.dense)
        return aligned32(xs) && aligned32(mm.dense) ? launch_worker<GT, false, true>(g, mm, xs, n, bits, scale, ws, st)
                                                    : launch_worker<GT, false, false>(g, mm, xs, n, bits, scale, ws, st);
    return aligned32(xs) ? launch_worker<GT, true, true>(g, mm, xs, n, bits, scale, ws, st)
                         : launch_worker<GT, true, false>(g, mm, xs, n, bits, scale, ws, st);
}

template <int PT>
int launch_update(const uint32_t *bits, const float *scales, int64_t S, int64_t n, int64_t numel, float *p,
                  float *m, const float *v, void *plp, void *ws, cudaStream_t st)
{
    const int64_t threads = n >> 3;
    const bool w32 = (!p || aligned32(p)) && (!v || aligned32(v)) && (!m || aligned32(m));
    auto kern = w32 ? k_onebit_update<PT, true> : k_onebit_update<PT, false>;
    launch_k(kern, (int)((threads + kThreads - 1) / kThreads), kThreads, st, false, bits, scales, S, n, numel, p, m,
             v, plp, (const StepScalars *)step_scalars(ws));
    return check_launch("zero_onebit_update");
}

}  // namespace
}  // namespace zpml

using namespace zpml;

extern "C" int zero_onebit_worker(const void *grad, int32_t gdtype, const float *m, const uint32_t *m_bits,
                                  const float *m_scales, int64_t S, float *x_w, int64_t n, uint32_t *bits,
                                  float *scale, const zero_hparams_t *hp, int64_t freeze_step,
                                  zero_state_t *d_state, void *ws, size_t ws_bytes, void *stream)
{
    if (!hp || !d_state || n < 0 || freeze_step < 1 || !hparams_ok(hp))
        return ZERO_EINVAL;
    if (!grad_dtype_ok(gdtype))
        return ZERO_EDTYPE;
    if (n % 32 != 0 || (n >> 3) / kThreads >= 0x7fffffff)
        return ZERO_ESIZE;
    if ((reinterpret_cast<uintptr_t>(d_state) & 7u) != 0)
        return ZERO_EALIGN;
    Momentum mm = {m, m_bits, m_scales, S};
    if (n > 0) {
        if (!grad || !x_w || !bits || !scale)
            return ZERO_EINVAL;
        if (!aligned16(grad) || !aligned16(x_w) || !aligned4(bits) || !aligned4(scale))
            return ZERO_EALIGN;
        if (!device_ptr(grad) || !device_ptr(x_w) || !device_ptr(bits) || !device_ptr(scale))
            return ZERO_EINVAL;
        if (m) {
            if (!aligned16(m))
                return ZERO_EALIGN;
            if (!device_ptr(m))
                return ZERO_EINVAL;
        } else {
            // the compressed momentum: S-element chunks, one scale each
            if (!m_bits || !m_scales || S <= 0)
                return ZERO_EINVAL;
            if (S % 32 != 0 || n % S != 0)
                return ZERO_ESIZE;
            if (!aligned4(m_bits) || !aligned4(m_scales))
                return ZERO_EALIGN;
            if (!device_ptr(m_bits) || !device_ptr(m_scales))
                return ZERO_EINVAL;
        }
    }
    if (!device_ptr(d_state))
        return ZERO_EINVAL;
    int rc = check_ws(ws, ws_bytes, 1, n);
    if (rc != ZERO_OK)
        return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const DecideArgs a = decide_args(hp, freeze_step);
    PowCache *cache = reinterpret_cast<PowCache *>(static_cast<unsigned char *>(ws) + kWsPowCache);
    // the decision also refills the bias-correction window: the 1-bit kernels
    // do not (its binary64 pow would raise their register counts)
    launch_k(k_decide, 1, 64, st, false, d_state, step_scalars(ws), cache, a, 1);
    if ((rc = check_launch("zero_onebit_worker (decision)")) != ZERO_OK || n == 0)
        return rc;
    switch (gdtype) {
    case ZERO_F16: return launch_worker_m<ZERO_F16>(grad, mm, x_w, n, bits, scale, ws, st);
    case ZERO_BF16: return launch_worker_m<ZERO_BF16>(grad, mm, x_w, n, bits, scale, ws, st);
    default: return launch_worker_m<ZERO_F32>(grad, mm, x_w, n, bits, scale, ws, st);
    }
}

extern "C" int zero_onebit_server(const uint32_t *const *worker_bits, const float *worker_scales, int32_t nd,
                                  int64_t S, float *x_s, uint32_t *bits, float *scale, void *ws, size_t ws_bytes,
                                  void *stream)
{
    if (nd < 1 || S < 0 || !worker_bits || !worker_scales)
        return ZERO_EINVAL;
    if (nd > kMaxServerWorkers)
        return ZERO_ECAPACITY;
    if (S % 32 != 0 || (S >> 3) / kThreads >= 0x7fffffff)
        return ZERO_ESIZE;
    for (int32_t k = 0; k < nd; ++k) {
        if (!worker_bits[k])
            return ZERO_EINVAL;
        if (!aligned4(worker_bits[k]))
            return ZERO_EALIGN;
    }
    if (!aligned4(worker_scales) || !device_ptr(worker_scales) || !device_ptr(worker_bits[0]) ||
        !device_ptr(worker_bits[nd - 1]))
        return !aligned4(worker_scales) ? ZERO_EALIGN : ZERO_EINVAL;
    if (S > 0) {
        if (!x_s || !bits || !scale)
            return ZERO_EINVAL;
        if (!aligned16(x_s) || !aligned4(bits) || !aligned4(scale))
            return ZERO_EALIGN;
        if (!device_ptr(x_s) || !device_ptr(bits) || !device_ptr(scale))
            return ZERO_EINVAL;
    }
    // up to kArgWorkers pointers go as a launch argument; more, as a table
    // in the workspace
    const bool by_arg = nd <= kArgWorkers;
    const size_t table = by_arg ? 0 : align256((size_t)nd * sizeof(void *));
    int rc = check_ws_table(ws, ws_bytes, table);
    if (rc != ZERO_OK)
        return rc;
    if (S == 0)
        return ZERO_OK;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    unsigned char *w = static_cast<unsigned char *>(ws);
    if (!by_arg) {
        std::vector<const uint32_t *> host(worker_bits, worker_bits + nd);
        rc = stage_upload(w + kWsTable, host.data(), (size_t)nd * sizeof(void *), st,
                          "zero_onebit_server (table upload)");
        if (rc != ZERO_OK)
            return rc;
    }
    const StepScalars *sc = step_scalars(ws);
    // persistent: two blocks per SM (each holds its own table), a warp per
    // 1024 elements at a time
    const int64_t warps = ((S >> 3) + 127) >> 7;
    int64_t grid = (int64_t)sm_count() * 2;
    if (grid > (warps + kWarps - 1) / kWarps)
        grid = (warps + kWarps - 1) / kWarps;
    if (grid > kMaxBlocks)
        grid = kMaxBlocks;
    if (grid < 1)
        grid = 1;
    const bool pow2 = (nd & (nd - 1)) == 0;
    const bool w32 = aligned32(x_s);
    const float inv_nd = pow2 ? 1.0f / (float)nd : 0.0f;  // exact: nd <= 2^12
    const size_t smem = server_smem_bytes(nd);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3((unsigned)kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    double2 *partials = reinterpret_cast<double2 *>(w + kWsPartials);
    WsHeader *hdr = reinterpret_cast<WsHeader *>(w);
    if (by_arg) {
        WorkerPtrs wp = {};
        for (int32_t k = 0; k < nd; ++k)
            wp.p[k] = worker_bits[k];
        auto kern = nd > 16 ? (pow2 ? (w32 ? k_onebit_server_args<true, true, true> : k_onebit_server_args<true, false, true>)
                                    : (w32 ? k_onebit_server_args<false, true, true> : k_onebit_server_args<false, false, true>))
                            : (pow2 ? (w32 ? k_onebit_server_args<true, true, false> : k_onebit_server_args<true, false, false>)
                                    : (w32 ? k_onebit_server_args<false, true, false> : k_onebit_server_args<false, false, false>));
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        cudaLaunchKernelEx(&cfg, kern, wp, worker_scales, (int)nd, inv_nd, x_s, S, sc, partials, hdr, scale, bits);
    } else {
        auto kern = pow2 ? (w32 ? k_onebit_server<true, true> : k_onebit_server<true, false>)
                         : (w32 ? k_onebit_server<false, true> : k_onebit_server<false, false>);
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        cudaLaunchKernelEx(&cfg, kern, (const uint32_t *const *)(w + kWsTable), worker_scales, (int)nd, inv_nd, x_s,
                           S, sc, partials, hdr, scale, bits);
    }
    return check_launch("zero_onebit_server");
}

extern "C" int zero_onebit_update(const uint32_t *bits, const float *server_scales, int32_t nd, int64_t S,
                                  int64_t numel, float *p, float *m, const float *v, void *p_lp, int32_t pdtype,
                                  void *ws, size_t ws_bytes, void *stream)
{
    if (nd < 1 || S < 0 || numel < 0 || !server_scales)
        return ZERO_EINVAL;
    if (S % 32 != 0 || S > ((int64_t)1 << 62) / nd || numel > (int64_t)nd * S ||
        (((int64_t)nd * S) >> 3) / kThreads >= 0x7fffffff)
        return ZERO_ESIZE;
    if (p_lp && !lp_dtype_ok(pdtype))
        return ZERO_EDTYPE;
    if ((int64_t)nd * S > 0) {
        if (!bits)
            return ZERO_EINVAL;
        if (!aligned4(bits) || !aligned4(server_scales) || (m && !aligned16(m)))
            return ZERO_EALIGN;
        if (!device_ptr(bits) || !device_ptr(server_scales) || (m && !device_ptr(m)))
            return ZERO_EINVAL;
    }
    if (numel > 0) {
        if (!p || !v)
            return ZERO_EINVAL;
        if (!aligned16(p) || !aligned16(v) || (p_lp && !aligned16(p_lp)))
            return ZERO_EALIGN;
        if (!device_ptr(p) || !device_ptr(v) || (p_lp && !device_ptr(p_lp)))
            return ZERO_EINVAL;
    }
    int rc = check_ws_table(ws, ws_bytes, 0);
    const int64_t n = (int64_t)nd * S;
    if (rc != ZERO_OK || n == 0)
        return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (!p_lp)
        return launch_update<kNoLowP>(bits, server_scales, S, n, numel, p, m, v, nullptr, ws, st);
    if (pdtype == ZERO_BF16)
        return launch_update<ZERO_BF16>(bits, server_scales, S, n, numel, p, m, v, p_lp, ws, st);
    return launch_update<ZERO_F16>(bits, server_scales, S, n, numel, p, m, v, p_lp, ws, st);
}
