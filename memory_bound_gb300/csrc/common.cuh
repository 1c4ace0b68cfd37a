// common.cuh -- device helpers shared by the fused-chain kernels (sm_103a).
//
// 16-byte fragments of fp32 / bf16 values, fp32 arithmetic helpers, warp and
// block reductions, and inline-PTX wrappers for mbarrier and bulk async copies
// (the Blackwell data-movement path used to stage rows into shared memory).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

namespace mb {

// Device-side failure bits (reported through mb_device_error).
constexpr unsigned kDevErrWaitTimeout = 1u;

// A barrier wait gives up after this many nanoseconds of %globaltimer (or this
// many polls, whichever comes first).  Real waits finish in microseconds.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;   // 2 s
constexpr unsigned kWaitLimitPolls = 1u << 28;

// ---------------------------------------------------------------------------
// programmatic dependent launch
// ---------------------------------------------------------------------------

// Waits until the grid this launch depends on (the previous kernel in the
// stream, when launched with programmatic stream serialisation) has completed
// and its memory is visible; returns at once otherwise.  Every kernel calls it
// before its first global memory access.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Lets the next kernel in the stream begin launching (its CTAs start as ours
// retire, and wait in pdl_wait for our completion).
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------------------
// scalar fp32 helpers
// ---------------------------------------------------------------------------

// relu with every value that is not > 0 (including -0 and NaN) mapped to +0.
__device__ __forceinline__ float relu_f(float v) { return v > 0.0f ? v : 0.0f; }

// 2^x and 1/x via the SFU (ex2.approx / rcp.approx, flush-to-zero).
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float rcp_approx(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// GeLU, tanh form, through the identity (1 + tanh(u)) / 2 = 1 / (1 + e^(-2u)):
//   gelu(n) = n / (1 + 2^(n * (c1 + c2 n^2)))
// with u = sqrt(2/pi) (n + 0.044715 n^3), c1 = -2 log2(e) sqrt(2/pi) and
// c2 = 0.044715 c1.  No 1 + tanh cancellation for n << 0; the limits are exact
// (2^t overflows to inf -> -0 for n << 0, underflows to 0 -> n for n >> 0).
__device__ __forceinline__ float gelu_tanh_f(float n) {
    constexpr double kSqrt2OverPi = 0.79788456080286535587989211986876;
    constexpr double kLog2e = 1.4426950408889634073599246810019;
    constexpr float c1 = (float)(-2.0 * kLog2e * kSqrt2OverPi);
    constexpr float c2 = (float)(-2.0 * kLog2e * kSqrt2OverPi * 0.044715);
    float n2 = n * n;
    float t = n * fmaf(c2, n2, c1);
    float e = ex2_approx(t);
    return n * rcp_approx(1.0f + e);
}

// The pointwise chain's four fp32 steps, each rounded on its own (no
// contraction), as the four eager ops round them.
__device__ __forceinline__ float add_relu_scale_1(float x, float b1, float b2, float scale) {
    float t = __fadd_rn(x, b1);       // x + b1
    t = relu_f(t);                    // relu
    t = __fmul_rn(t, scale);          // * scale
    return __fadd_rn(t, b2);          // + b2
}

// Pairs of fp32 values through Blackwell's packed fp32x2 instructions: each
// lane is an ordinary IEEE fp32 operation rounded to nearest, so results are
// the same as two scalar operations, at half the instruction issue.
__device__ __forceinline__ float2 add2(float2 a, float2 b) { return __fadd2_rn(a, b); }
__device__ __forceinline__ float2 mul2(float2 a, float2 b) { return __fmul2_rn(a, b); }
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }
__device__ __forceinline__ float2 splat2(float a) { return make_float2(a, a); }
__device__ __forceinline__ float2 relu2(float2 a) { return make_float2(relu_f(a.x), relu_f(a.y)); }

// ---------------------------------------------------------------------------
// counter-based random numbers for dropout
// ---------------------------------------------------------------------------

// Philox-4x32-10 ("Parallel random numbers: as easy as 1, 2, 3", Salmon,
// Moraes, Dror and Shaw, SC'11): ten rounds over a 4-word counter; each round
// takes the full 64-bit products of words 0 and 2 with the two multipliers and
// forms (hi(M1 c2) ^ c1 ^ k0, lo(M1 c2), hi(M0 c0) ^ c3 ^ k1, lo(M0 c0)),
// with the key bumped by the Weyl constants (golden ratio and sqrt(3) - 1)
// before every round but the first.
constexpr uint32_t kPhiloxM0 = 0xD2511F53u, kPhiloxM1 = 0xCD9E8D57u;
constexpr uint32_t kPhiloxW0 = 0x9E3779B9u, kPhiloxW1 = 0xBB67AE85u;

// Dropout parameters, prepared on the host.  The round keys are the key
// schedule written out (rk[2r], rk[2r + 1] = key + r (W0, W1)), so the kernel
// reads them as launch constants.  One block serves eight elements: element i
// takes the 16-bit half (i mod 2: low, high) of word (i mod 8) / 2 of the block
// at counter (0, 0, lo(g), hi(g)), g = offset + i / 8, and is kept iff that
// half, as a fraction of 2^16, is >= p: iff half >= thr = ceil(p 2^16) (the
// same decision, taken exactly in integers).  Kept values are scaled by
// inv_keep = 1 / (1 - p); dropped ones are multiplied by 0.
struct DropoutArgs {
    uint32_t rk[20];
    uint64_t offset;
    uint32_t thr;
    float inv_keep;
};

// The block at counter (0, 0, lo(g), hi(g)).
__device__ __forceinline__ uint4 philox_block(uint64_t g, const DropoutArgs &d) {
    uint32_t c0 = 0u, c1 = 0u, c2 = (uint32_t)g, c3 = (uint32_t)(g >> 32);
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        const uint32_t hi0 = __umulhi(kPhiloxM0, c0), lo0 = kPhiloxM0 * c0;
        const uint32_t hi1 = __umulhi(kPhiloxM1, c2), lo1 = kPhiloxM1 * c2;
        c0 = hi1 ^ c1 ^ d.rk[2 * r];
        c1 = lo1;
        c2 = hi0 ^ c3 ^ d.rk[2 * r + 1];
        c3 = lo0;
    }
    return make_uint4(c0, c1, c2, c3);
}

__device__ __forceinline__ float keep_scale(uint32_t half, const DropoutArgs &d) {
    return half >= d.thr ? d.inv_keep : 0.0f;
}

// The keep decisions of the eight elements of block g, as bits (bit e: the
// element of index 8 (g - offset) + e is kept).
__device__ __forceinline__ uint32_t keep_bits8(uint64_t g, const DropoutArgs &d) {
    const uint4 w = philox_block(g, d);
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
    uint32_t m = 0u;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        m |= (uint32_t)((ws[k] & 0xFFFFu) >= d.thr) << (2 * k);
        m |= (uint32_t)((ws[k] >> 16) >= d.thr) << (2 * k + 1);
    }
    return m;
}

// The dropout draws of one slot of VEC elements.  A slot of eight or more
// keeps its keep decisions as bits (bit e: element e of the slot); a scalar
// slot keeps its element's 16-bit half.
template <int VEC> struct DropBits {
    static constexpr bool kMask = VEC % 8 == 0;
    static constexpr int kWords = kMask ? 1 : VEC;
    uint32_t w[kWords];
};

// The draws of the slot whose first element has index `off` in the whole
// tensor (they depend on nothing else, so they can be drawn early).  A slot
// of eight elements starts on a block (off a multiple of 8) on the aligned
// engines; with ANYOFF (the shifted-vector engine) it may start at s = off
// mod 8 > 0 and then spans blocks off / 8 and the next one: their sixteen
// keep bits shifted down by s (s is the same for every slot of a row, so the
// branch is uniform).
template <int VEC, bool ANYOFF = false>
__device__ __forceinline__ void dropout_bits(int64_t off, const DropoutArgs &d, DropBits<VEC> &b) {
    if constexpr (VEC % 8 == 0) {
        const uint64_t g0 = d.offset + (uint64_t)(off >> 3);
        uint32_t m = 0u;
#pragma unroll
        for (int q = 0; q < VEC / 8; ++q) {
            uint32_t bits = keep_bits8(g0 + (uint64_t)q, d);
            if constexpr (ANYOFF) {
                const int sh = (int)(off & 7);
                if (sh) bits = (bits | keep_bits8(g0 + (uint64_t)q + 1u, d) << 8) >> sh;
            }
            m |= (bits & 0xFFu) << (8 * q);
        }
        b.w[0] = m;
    } else {
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
            const int64_t i = off + e;
            const uint4 w = philox_block(d.offset + (uint64_t)(i >> 3), d);
            const int k = (int)((i & 7) >> 1);
            const uint32_t word = k == 0 ? w.x : k == 1 ? w.y : k == 2 ? w.z : w.w;
            b.w[e] = (i & 1) ? (word >> 16) : (word & 0xFFFFu);
        }
    }
}

// Applies the decisions: kept values times 1 / (1 - p), dropped ones times 0.
template <int VEC>
__device__ __forceinline__ void dropout_apply(float (&o)[VEC], const DropBits<VEC> &b,
                                              const DropoutArgs &d) {
    if constexpr (VEC % 8 == 0) {
#pragma unroll
        for (int e = 0; e < VEC; ++e) o[e] *= ((b.w[0] >> e) & 1u) ? d.inv_keep : 0.0f;
    } else {
#pragma unroll
        for (int e = 0; e < VEC; ++e) o[e] *= keep_scale(b.w[e], d);
    }
}

// ---------------------------------------------------------------------------
// bf16 packing (raw 16-bit patterns, little-endian pairs in 32-bit words)
// ---------------------------------------------------------------------------

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);   // round to nearest even
    return *reinterpret_cast<uint32_t *>(&h);
}
__device__ __forceinline__ float bf16_to_f(uint16_t h) { return __uint_as_float((uint32_t)h << 16); }
__device__ __forceinline__ uint16_t f_to_bf16(float f) {
    __nv_bfloat16 h = __float2bfloat16_rn(f);
    return *reinterpret_cast<uint16_t *>(&h);
}

// ---------------------------------------------------------------------------
// Fragments: VEC consecutive elements of one tensor as fp32 values.
// VEC * sizeof(T) a multiple of 16 uses that many 128-bit accesses; VEC == 1
// is a scalar access.  T is float or uint16_t (bf16 bits).
// ---------------------------------------------------------------------------

template <typename T> struct Elem;
template <> struct Elem<float> { static constexpr int kVec = 4; };
template <> struct Elem<uint16_t> { static constexpr int kVec = 8; };

template <typename T, int VEC> struct Frag {
    // 16-byte accesses per fragment (0: one scalar access)
    static constexpr int kParts = VEC * (int)sizeof(T) / 16;
    static constexpr int kPer = 16 / (int)sizeof(T);    // elements per 16 bytes
    static_assert(VEC == 1 || (kParts >= 1 && kParts * kPer == VEC), "fragment size");
    float f[VEC];

    // elements [q * kPer, (q + 1) * kPer) from / to one 16-byte word
    __device__ __forceinline__ void unpack(const uint4 &u, int q) {
        float *g = f + q * kPer;
        if constexpr (sizeof(T) == 4) {
            g[0] = __uint_as_float(u.x); g[1] = __uint_as_float(u.y);
            g[2] = __uint_as_float(u.z); g[3] = __uint_as_float(u.w);
        } else {
            g[0] = bf16_lo(u.x); g[1] = bf16_hi(u.x);
            g[2] = bf16_lo(u.y); g[3] = bf16_hi(u.y);
            g[4] = bf16_lo(u.z); g[5] = bf16_hi(u.z);
            g[6] = bf16_lo(u.w); g[7] = bf16_hi(u.w);
        }
    }
    __device__ __forceinline__ uint4 pack(int q) const {
        const float *g = f + q * kPer;
        uint4 u;
        if constexpr (sizeof(T) == 4) {
            u.x = __float_as_uint(g[0]); u.y = __float_as_uint(g[1]);
            u.z = __float_as_uint(g[2]); u.w = __float_as_uint(g[3]);
        } else {
            u.x = pack_bf16x2(g[0], g[1]); u.y = pack_bf16x2(g[2], g[3]);
            u.z = pack_bf16x2(g[4], g[5]); u.w = pack_bf16x2(g[6], g[7]);
        }
        return u;
    }
    __device__ __forceinline__ static float to_f(T v) {
        if constexpr (sizeof(T) == 4) return v; else return bf16_to_f(v);
    }
    __device__ __forceinline__ static T from_f(float v) {
        if constexpr (sizeof(T) == 4) return v; else return f_to_bf16(v);
    }

    // streaming load of row data (evict-first in cache)
    __device__ __forceinline__ void load_stream(const T *p) {
        if constexpr (VEC == 1) {
            f[0] = to_f(__ldcs(p));
        } else {
#pragma unroll
            for (int q = 0; q < kParts; ++q)
                unpack(__ldcs(reinterpret_cast<const uint4 *>(p) + q), q);
        }
    }
    // the streaming load when `take`, else zeros (a slot the chain never
    // reads: the masked tail of a causal score row)
    __device__ __forceinline__ void load_stream_if(const T *p, bool take) {
        if (take) {
            load_stream(p);
        } else {
#pragma unroll
            for (int e = 0; e < VEC; ++e) f[e] = 0.0f;
        }
    }
    // cached read-only load (per-column vectors, reused by every row)
    __device__ __forceinline__ void load_cached(const T *p) {
        if constexpr (VEC == 1) {
            f[0] = to_f(__ldg(p));
        } else {
#pragma unroll
            for (int q = 0; q < kParts; ++q)
                unpack(__ldg(reinterpret_cast<const uint4 *>(p) + q), q);
        }
    }
    // the cached load element by element, for per-column values whose
    // columns do not start on a 16-byte boundary
    __device__ __forceinline__ void load_cached_elems(const T *p) {
#pragma unroll
        for (int e = 0; e < VEC; ++e) f[e] = to_f(__ldg(p + e));
    }
    // load_cached when AL (16-byte aligned columns), else load_cached_elems
    template <bool AL> __device__ __forceinline__ void load_cached_as(const T *p) {
        if constexpr (AL) load_cached(p); else load_cached_elems(p);
    }
    __device__ __forceinline__ void load_shared(const T *p) {
        if constexpr (VEC == 1) {
            f[0] = to_f(*p);
        } else {
#pragma unroll
            for (int q = 0; q < kParts; ++q) unpack(reinterpret_cast<const uint4 *>(p)[q], q);
        }
    }
    __device__ __forceinline__ void store_stream(T *p) const {
        if constexpr (VEC == 1) {
            __stcs(p, from_f(f[0]));
        } else {
#pragma unroll
            for (int q = 0; q < kParts; ++q) __stcs(reinterpret_cast<uint4 *>(p) + q, pack(q));
        }
    }
};

// Where a vector slot's per-column values come from (the chains' load_pre /
// load_post hooks take one; `i` numbers the chain's per-column arrays).
// ColsGlobal: the arrays in global memory through the read-only cache, one
// 16-byte access per 16 bytes when AL (the slot's columns start on a 16-byte
// boundary), else element by element.
template <bool AL> struct ColsGlobal {
    template <typename T, int VEC>
    __device__ __forceinline__ void operator()(Frag<T, VEC> &f, const T *arr, int col,
                                               int) const {
        f.template load_cached_as<AL>(arr + col);
    }
};
// ColsShared: the CTA's copy of every per-column array in shared memory,
// starting at column h: array i's column c sits at s[i * stride + c - h], so a
// slot whose columns start at h + k * VEC is one 16-byte aligned access when
// s and stride * sizeof(T) are multiples of 16 bytes.
template <typename T> struct ColsShared {
    const T *s;
    int stride;
    int h;
    template <int VEC>
    __device__ __forceinline__ void operator()(Frag<T, VEC> &f, const T *, int col, int i) const {
        f.load_shared(s + i * stride + (col - h));
    }
};

// ---------------------------------------------------------------------------
// reductions (every lane / thread ends with the bitwise-same value)
// ---------------------------------------------------------------------------

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
    return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, m));
    return v;
}

// Maximum over the CTA; same buffer discipline as block_sum below.
__device__ __forceinline__ float block_max(float v, float *red) {
    v = warp_max(v);
    const int lane = threadIdx.x & 31;
    if (lane == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    return warp_max(lane < (int)(blockDim.x >> 5) ? red[lane] : -INFINITY);
}

// Sum over the CTA.  `red` holds 32 floats of shared memory; callers alternate
// between two such buffers so that one reduction's reads cannot race with the
// next one's writes.  After the barrier every warp runs the same butterfly
// over the per-warp partials (lane i holds partial i, zero past the last
// warp), so all threads get the bitwise-same result.
__device__ __forceinline__ float block_sum(float v, float *red) {
    v = warp_sum(v);
    const int lane = threadIdx.x & 31;
    if (lane == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    return warp_sum(lane < (int)(blockDim.x >> 5) ? red[lane] : 0.0f);
}

// ---------------------------------------------------------------------------
// mbarrier + bulk async copy (global -> shared), inline PTX
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Make barrier initialisation visible to the async proxy.
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

// One bulk copy of `bytes` (multiple of 16; both addresses 16-byte aligned)
// from global to shared memory, completing on `bar` as transaction bytes.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes,
                                         uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(__cvta_generic_to_global(src)), "r"(bytes), "r"(bar)
        : "memory");
}

// One 4-byte asynchronous copy from global to shared memory (both addresses
// 4-byte aligned); it is complete for the issuing thread after cp_async_wait_all.
__device__ __forceinline__ void cp_async4(uint32_t dst, const void *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst),
                 "l"(__cvta_generic_to_global(src))
                 : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.wait_all;" ::: "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ unsigned long long globaltimer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Arrive on a local mbarrier and add `bytes` to the transaction count it
// expects, with no release of this thread's earlier accesses (so loads and
// stores still in flight do not have to land first).
__device__ __forceinline__ void mbar_arrive_expect_tx_relaxed(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.relaxed.cta.shared::cta.b64 _, [%0], %1;"
                 :: "r"(bar), "r"(bytes) : "memory");
}

// The address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_cluster(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

// Stores 4 bytes into another CTA's shared memory (a cluster address) and
// completes 4 transaction bytes on that CTA's mbarrier `remote_bar`.
__device__ __forceinline__ void st_async_f32(uint32_t remote_addr, float v, uint32_t remote_bar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];"
                 :: "r"(remote_addr), "r"(__float_as_uint(v)), "r"(remote_bar) : "memory");
}

// Wait for phase `parity` of `bar` to complete, giving up after `limit_ns`
// of %globaltimer (or kWaitLimitPolls polls).  Returns false if it gave up.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  unsigned long long limit_ns = kWaitLimitNs) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer_ns();
    for (unsigned i = 0; i < kWaitLimitPolls; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 15u) == 15u && globaltimer_ns() - t0 > limit_ns) return false;
    }
    return false;
}

}  // namespace mb
