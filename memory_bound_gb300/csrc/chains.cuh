// chains.cuh -- the per-element arithmetic of the reduce-plus-pointwise
// chains, plugged into the row engines of rows.cuh.
//
// Every hook works on one slot of VEC values of a row.  Vector slots (VEC 4
// or 8) run their arithmetic in pairs through the packed fp32x2 instructions
// (add2 / mul2 / fma2: per lane the same IEEE fp32 operation, rounded to
// nearest, as the scalar form); scalar slots (VEC 1) use the scalar forms.
#pragma once

#include <type_traits>

#include "rows.cuh"

namespace mb {

// Per-slot values a chain draws before the row arrives (hook `early`), for
// chains that have none.
struct NoEarly {};

// v <- v - s for a slot; returns the sum of the squares (second LN pass)
template <int VEC>
__device__ __forceinline__ float center_sumsq(float (&v)[VEC], float s) {
    if constexpr (VEC == 1) {
        v[0] = v[0] - s;
        return v[0] * v[0];
    } else {
        float2 acc = splat2(0.0f);
#pragma unroll
        for (int e = 0; e < VEC; e += 2) {
            const float2 d = add2(make_float2(v[e], v[e + 1]), splat2(-s));
            v[e] = d.x;
            v[e + 1] = d.y;
            acc = fma2(d, d, acc);
        }
        return acc.x + acc.y;
    }
}

// o = act(v * rstd * w + b) for a slot of centred values (LayerNorm epilogue)
template <typename T, int VEC, int ACT>
__device__ __forceinline__ void ln_affine_act(const float (&v)[VEC], float rstd,
                                              const Frag<T, VEC> &w, const Frag<T, VEC> &b,
                                              float (&o)[VEC]) {
    if constexpr (VEC == 1) {
        const float n = fmaf(v[0] * rstd, w.f[0], b.f[0]);
        o[0] = ACT == 2 ? gelu_tanh_f(n) : (ACT == 1 ? relu_f(n) : n);
    } else if constexpr (ACT == 2) {
        // scalar here: measured 0.8% faster on the bf16 LN workload than the
        // paired form (the pair shuffling costs about what it saves)
#pragma unroll
        for (int e = 0; e < VEC; ++e) o[e] = gelu_tanh_f(fmaf(v[e] * rstd, w.f[e], b.f[e]));
    } else {
#pragma unroll
        for (int e = 0; e < VEC; e += 2) {
            const float2 xh = mul2(make_float2(v[e], v[e + 1]), splat2(rstd));
            float2 n = fma2(xh, make_float2(w.f[e], w.f[e + 1]), make_float2(b.f[e], b.f[e + 1]));
            if constexpr (ACT == 1) n = relu2(n);
            o[e] = n.x;
            o[e + 1] = n.y;
        }
    }
}

// v = x + r for a slot
template <typename T, int VEC>
__device__ __forceinline__ void add_inputs(const Frag<T, VEC> &x, const Frag<T, VEC> &r,
                                           float (&v)[VEC]) {
    if constexpr (VEC == 1) {
        v[0] = __fadd_rn(x.f[0], r.f[0]);
    } else {
#pragma unroll
        for (int e = 0; e < VEC; e += 2) {
            const float2 s = add2(make_float2(x.f[e], x.f[e + 1]), make_float2(r.f[e], r.f[e + 1]));
            v[e] = s.x;
            v[e + 1] = s.y;
        }
    }
}

// Residual + LayerNorm + affine + GeLU-tanh.
// "Operator fusion and kernel optimisation" (plumephp.com) §2.2-2.3: v = x +
// residual, row mean and variance, rsqrt(var + eps), (v - mean) * inv_std *
// weight + bias, then GeLU (tanh form).  "Kernel fusion" course chapter 4
// (5688vip.com) §4.3: the variance as a second pass, sum((v - mean)^2) / cols.
template <typename TT> struct LnGeluChain {
    using T = TT;
    static constexpr int kInputs = 2;     // x, r
    static constexpr int kVec = Elem<T>::kVec;   // elements per vector slot (16 bytes)
    static constexpr bool kRegCap = false;     // see LnActChain
    static constexpr int kRowsTarget = 0;
    static constexpr int kWideScalarSlots = 32;   // see LnActChain
    static constexpr bool kShiftOk = true;        // see LnActChain
    // values per thread the cluster planner prefers for rows longer than a
    // CTA: 16 for fp32 (x, r, w and b held per value; 32 ran LN at 65536
    // columns 5% slower), 32 for bf16 rows (3% faster than 16)
    static constexpr int kClusterVals = sizeof(T) == 2 ? 32 : 16;
    static constexpr bool kStageLargeSlices = false;   // measured slower staged
    static constexpr bool kPartialRows = false;   // every row read whole
    static constexpr bool kTwoPass = true;
    static constexpr bool kMaxFirst = false;
    static constexpr bool kStorePre = false;
    struct Args {
        const T *in[2];
        const T *w;
        const T *b;
        T *out;
        float eps;
        float inv_cols;   // 1 / H, rounded to fp32 on the host
    };
    // per-column values of one slot: none before the reduction, w and b after
    template <int VEC> struct PrePC {};
    template <int VEC> struct PostPC { Frag<T, VEC> w, b; };
    static constexpr int kPostPC = 2;     // per-column vectors the epilogue reads
    // the per-column arrays, numbered as the load hooks number them
    static constexpr int kColArrays = 2;
    __host__ __device__ __forceinline__ static const T *col_array(const Args &a, int i) {
        return i == 0 ? a.w : a.b;
    }
    // rows off the 16-byte grid may take the shifted kernel's staged form
    static constexpr bool kShiftStaged = true;
    template <int VEC> using Early = NoEarly;
    template <int VEC, bool ANYOFF = false>
    __device__ __forceinline__ static void early(const Args &, int64_t, Early<VEC> &) {}
    template <int VEC, class LD = ColsGlobal<true>>
    __device__ __forceinline__ static void load_pre(const Args &, int, PrePC<VEC> &,
                                                    const LD & = LD{}) {}
    template <int VEC, class LD = ColsGlobal<true>>
    __device__ __forceinline__ static void load_post(const Args &a, int col, PostPC<VEC> &pc,
                                                     const LD &ld = LD{}) {
        ld(pc.w, a.w, col, 0);
        ld(pc.b, a.b, col, 1);
    }
    template <int VEC>
    __device__ __forceinline__ static void pre(const Frag<T, VEC> (&in)[2], const PrePC<VEC> &,
                                               const Args &, int64_t, int, float (&v)[VEC]) {
        add_inputs<T, VEC>(in[0], in[1], v);
    }
    template <int VEC>
    __device__ __forceinline__ static void store_pre(const float (&)[VEC], const Args &, int64_t) {}
    // mean = sum(v) / H; second pass: v <- v - mean, summing the squares;
    // rstd = 1/sqrt(var + eps)
    // mean = sum * (1 / H), the reciprocal a launch argument (exact for H a
    // power of 2): an operand read from the parameter bank, so it takes no
    // register across the row loop (a reciprocal hoisted out of the loop by
    // the compiler did, and pushed the 1024-thread cluster kernel into spills)
    __device__ __forceinline__ static float stat1(float sum, int, const Args &a) {
        return sum * a.inv_cols;
    }
    template <int VEC>
    __device__ __forceinline__ static float p2(float (&v)[VEC], float mean) {
        return center_sumsq<VEC>(v, mean);
    }
    __device__ __forceinline__ static float stat2(float m2, int, const Args &a) {
        return rsqrtf(m2 * a.inv_cols + a.eps);
    }
    __device__ __forceinline__ static void store_stats(const Args &, int64_t, float, float) {}
    static int outputs(const Args &) { return 1; }
    static int read_percent(const Args &, int64_t, int) { return 100; }
    // leading elements of row `row` the chain reads (the staged engines copy no more)
    __host__ __device__ static int row_extent(const Args &, int64_t, int cols) { return cols; }
    template <int VEC>
    __device__ __forceinline__ static void post(const float (&v)[VEC], float, float rstd,
                                                const PostPC<VEC> &pc, const Args &, int64_t,
                                                const Early<VEC> &, float (&o)[VEC]) {
        ln_affine_act<T, VEC, 2>(v, rstd, pc.w, pc.b, o);
    }
};

// TorchInductor example chain ("TorchInductor Pipeline and operator fusion",
// blog.kkkzoz.top, the example model and Figure 1):
//   t = x * x_scale + bias; a = relu(t); p = a * a; q = a * branch_scale;
//   s = p + q; m = mean(s, dim=1); y = (s - m) * gamma + beta.
// Each pointwise step is rounded on its own (no contraction), as the fp32
// eager ops would round it; s is recomputed in registers, never stored, and
// the row sum never leaves the chip (§08 of the same post).  With bf16 I/O
// the inputs are widened exactly and y is rounded once.
template <typename TT> struct InductorChainT {
    using T = TT;
    static constexpr int kInputs = 1;     // x
    static constexpr int kVec = Elem<T>::kVec;
    static constexpr bool kRegCap = false;     // see LnActChain
    static constexpr int kRowsTarget = 0;
    static constexpr int kWideScalarSlots = 32;   // see LnActChain
    static constexpr bool kShiftOk = true;        // see LnActChain
    static constexpr int kClusterVals = 16;   // see LnGeluChain
    static constexpr bool kStageLargeSlices = false;   // measured slower staged
    static constexpr bool kPartialRows = false;   // every row read whole
    static constexpr bool kTwoPass = false;
    static constexpr bool kMaxFirst = false;
    static constexpr bool kStorePre = false;
    struct Args {
        const T *in[1];
        const T *bias;
        const T *gamma;
        const T *beta;
        T *out;
        float x_scale;
        float branch_scale;
    };
    // per-column values of one slot: bias before the reduction, gamma and beta after
    template <int VEC> struct PrePC { Frag<T, VEC> bias; };
    template <int VEC> struct PostPC { Frag<T, VEC> gamma, beta; };
    static constexpr int kPostPC = 2;
    static constexpr int kColArrays = 3;      // bias, gamma, beta (see LnGeluChain)
    __host__ __device__ __forceinline__ static const T *col_array(const Args &a, int i) {
        return i == 0 ? a.bias : i == 1 ? a.gamma : a.beta;
    }
    static constexpr bool kShiftStaged = true;    // see LnGeluChain
    template <int VEC> using Early = NoEarly;
    template <int VEC, bool ANYOFF = false>
    __device__ __forceinline__ static void early(const Args &, int64_t, Early<VEC> &) {}
    template <int VEC, class LD = ColsGlobal<true>>
    __device__ __forceinline__ static void load_pre(const Args &a, int col, PrePC<VEC> &pc,
                                                    const LD &ld = LD{}) {
        ld(pc.bias, a.bias, col, 0);
    }
    template <int VEC, class LD = ColsGlobal<true>>
    __device__ __forceinline__ static void load_post(const Args &a, int col, PostPC<VEC> &pc,
                                                     const LD &ld = LD{}) {
        ld(pc.gamma, a.gamma, col, 1);
        ld(pc.beta, a.beta, col, 2);
    }
    template <int VEC>
    __device__ __forceinline__ static void pre(const Frag<T, VEC> (&in)[1],
                                               const PrePC<VEC> &pc, const Args &a, int64_t, int,
                                               float (&v)[VEC]) {
        if constexpr (VEC == 1) {
            const float t = __fadd_rn(__fmul_rn(in[0].f[0], a.x_scale), pc.bias.f[0]);
            const float r = relu_f(t);
            v[0] = __fadd_rn(__fmul_rn(r, r), __fmul_rn(r, a.branch_scale));
        } else {
#pragma unroll
            for (int e = 0; e < VEC; e += 2) {
                const float2 t = add2(mul2(make_float2(in[0].f[e], in[0].f[e + 1]), splat2(a.x_scale)),
                                      make_float2(pc.bias.f[e], pc.bias.f[e + 1]));
                const float2 r = relu2(t);
                const float2 s = add2(mul2(r, r), mul2(r, splat2(a.branch_scale)));
                v[e] = s.x;
                v[e + 1] = s.y;
            }
        }
    }
    template <int VEC>
    __device__ __forceinline__ static void store_pre(const float (&)[VEC], const Args &, int64_t) {}
    // m = sum(s) / cols (a row sum divided by the row length); no second pass
    __device__ __forceinline__ static float stat1(float sum, int cols, const Args &) {
        return sum / (float)cols;
    }
    template <int VEC>
    __device__ __forceinline__ static float p2(float (&)[VEC], float) { return 0.0f; }
    __device__ __forceinline__ static float stat2(float, int, const Args &) { return 0.0f; }
    __device__ __forceinline__ static void store_stats(const Args &, int64_t, float, float) {}
    static int outputs(const Args &) { return 1; }
    static int read_percent(const Args &, int64_t, int) { return 100; }
    // leading elements of row `row` the chain reads (the staged engines copy no more)
    __host__ __device__ static int row_extent(const Args &, int64_t, int cols) { return cols; }
    template <int VEC>
    __device__ __forceinline__ static void post(const float (&v)[VEC], float mean, float,
                                                const PostPC<VEC> &pc, const Args &, int64_t,
                                                const Early<VEC> &, float (&o)[VEC]) {
        if constexpr (VEC == 1) {
            o[0] = __fadd_rn(__fmul_rn(__fsub_rn(v[0], mean), pc.gamma.f[0]), pc.beta.f[0]);
        } else {
#pragma unroll
            for (int e = 0; e < VEC; e += 2) {
                // s - m as s + (-m): the same rounding
                const float2 d = add2(make_float2(v[e], v[e + 1]), splat2(-mean));
                const float2 y = add2(mul2(d, make_float2(pc.gamma.f[e], pc.gamma.f[e + 1])),
                                      make_float2(pc.beta.f[e], pc.beta.f[e + 1]));
                o[e] = y.x;
                o[e + 1] = y.y;
            }
        }
    }
};
using InductorChain = InductorChainT<float>;

// LayerNorm family: v = x (+ r); optionally h = v written out (the residual
// stream); out = act((v - mean) * rstd * w + b), act none / relu / gelu-tanh;
// with DROP, dropout on out (§2.1 of the same page: LayerNorm -> ReLU ->
// Dropout in one kernel); optionally the per-row mean and rstd written out.
// "Kernel fusion" course chapter 4 (5688vip.com) §4.3 (LayerNorm, two-pass
// variance); "Operator fusion and kernel optimisation" (plumephp.com) §2.1
// (LayerNorm -> ReLU in one kernel) and §2.2-2.3 (residual + LayerNorm + GeLU).
enum { kActNone = 0, kActRelu = 1, kActGelu = 2 };
template <typename TT, bool RES, bool DROP = false> struct LnActChain {
    using T = TT;
    static constexpr int kInputs = RES ? 2 : 1;
    // with dropout a slot is eight elements (one generator block; 32 bytes
    // of fp32), else 16 bytes
    static constexpr int kVec = DROP ? 8 : Elem<T>::kVec;
    // With dropout on fp32 rows the kernel is latency-bound (the generator's
    // multiply chains): registers capped (rows_cta_kernel_capped) so that six
    // 256-thread CTAs share an SM, and six rows in flight per SM.  Measured
    // on GB300 (8192 x 4096 fp32): 49.4 us against 51.2 uncapped with four.
    // bf16 rows hold twice the values per byte and would spill under the cap,
    // and the cap slows the other chains (LN bf16 245 -> 296 us): they keep
    // the ordinary kernel.
    static constexpr bool kRegCap = DROP && sizeof(T) == 4;
    static constexpr int kRowsTarget = kRegCap ? 6 : 0;
    // scalar slots per thread from which the one-CTA engine takes its
    // 512-thread form (the 1024-thread one spills from there on)
    static constexpr int kWideScalarSlots = DROP ? 16 : 32;
    // rows off the 16-byte grid may take the shifted-vector engine (with
    // dropout, a slot may start anywhere within a block of eight: its keep
    // bits come from one or two blocks, dropout_bits)
    static constexpr bool kShiftOk = true;
    static constexpr int kClusterVals = sizeof(T) == 2 ? 32 : 16;   // as LnGeluChain
    static constexpr bool kStageLargeSlices = false;   // measured slower staged
    static constexpr bool kPartialRows = false;   // every row read whole
    static constexpr bool kTwoPass = true;
    static constexpr bool kMaxFirst = false;
    static constexpr bool kStorePre = true;
    struct Args {
        const T *in[kInputs];
        const T *w;
        const T *b;
        T *out;
        T *h;          // residual-stream output (NULL: not written)
        float eps;
        int act;
        float *mean_out;   // per-row mean (NULL: not written)
        float *rstd_out;   // per-row 1/sqrt(var + eps) (NULL: not written)
        DropoutArgs drop;  // used with DROP only
        float inv_cols;    // 1 / H, rounded to fp32 on the host
    };
    template <int VEC> struct PrePC {};
    template <int VEC> struct PostPC { Frag<T, VEC> w, b; };
    static constexpr int kPostPC = 2;
    static constexpr int kColArrays = 2;      // w, b (see LnGeluChain)
    __host__ __device__ __forceinline__ static const T *col_array(const Args &a, int i) {
        return i == 0 ? a.w : a.b;
    }
    // With dropout the shifted rows keep the unstaged form: the generator
    // keeps those kernels issue-bound, and the staged form ran 1-10% slower
    // (fp32 rows of 2051-12291, bf16 of 4099 and 8195).
    static constexpr bool kShiftStaged = !DROP;
    // with dropout: the slot's 16-bit uniforms, drawn while the row is in
    // flight (they depend only on the element index)
    template <int VEC> struct EarlyDrop { DropBits<VEC> bits; };
    template <int VEC> using Early = std::conditional_t<DROP, EarlyDrop<VEC>, NoEarly>;
    template <int VEC, bool ANYOFF = false>
    __device__ __forceinline__ static void early(const Args &a, int64_t off, Early<VEC> &e) {
        if constexpr (DROP) dropout_bits<VEC, ANYOFF>(off, a.drop, e.bits);
    }
    template <int VEC, class LD = ColsGlobal<true>>
    __device__ __forceinline__ static void load_pre(const Args &, int, PrePC<VEC> &,
                                                    const LD & = LD{}) {}
    template <int VEC, class LD = ColsGlobal<true>>
    __device__ __forceinline__ static void load_post(const Args &a, int col, PostPC<VEC> &pc,
                                                     const LD &ld = LD{}) {
        ld(pc.w, a.w, col, 0);
        ld(pc.b, a.b, col, 1);
    }
    template <int VEC>
    __device__ __forceinline__ static void pre(const Frag<T, VEC> (&in)[kInputs],
                                               const PrePC<VEC> &, const Args &, int64_t, int,
                                               float (&v)[VEC]) {
        if constexpr (RES) {
            add_inputs<T, VEC>(in[0], in[1], v);
        } else {
#pragma unroll
            for (int e = 0; e < VEC; ++e) v[e] = in[0].f[e];
        }
    }
    template <int VEC>
    __device__ __forceinline__ static void store_pre(const float (&v)[VEC], const Args &a,
                                                     int64_t off) {
        if (a.h) {
            Frag<T, VEC> f;
#pragma unroll
            for (int e = 0; e < VEC; ++e) f.f[e] = v[e];
            f.store_stream(a.h + off);
        }
    }
    // mean = sum * (1 / H), the reciprocal a launch argument (as in LnGeluChain)
    __device__ __forceinline__ static float stat1(float sum, int, const Args &a) {
        return sum * a.inv_cols;
    }
    template <int VEC>
    __device__ __forceinline__ static float p2(float (&v)[VEC], float mean) {
        return center_sumsq<VEC>(v, mean);
    }
    __device__ __forceinline__ static float stat2(float m2, int, const Args &a) {
        return rsqrtf(m2 * a.inv_cols + a.eps);
    }
    template <int VEC>
    __device__ __forceinline__ static void post(const float (&v)[VEC], float, float rstd,
                                                const PostPC<VEC> &pc, const Args &a,
                                                int64_t, const Early<VEC> &ea,
                                                float (&o)[VEC]) {
        if (a.act == kActGelu) ln_affine_act<T, VEC, 2>(v, rstd, pc.w, pc.b, o);
        else if (a.act == kActRelu) ln_affine_act<T, VEC, 1>(v, rstd, pc.w, pc.b, o);
        else ln_affine_act<T, VEC, 0>(v, rstd, pc.w, pc.b, o);
        if constexpr (DROP) dropout_apply<VEC>(o, ea.bits, a.drop);
    }
    // full-size outputs per row: out, and h when it is written
    static int outputs(const Args &a) { return a.h ? 2 : 1; }
    static int read_percent(const Args &, int64_t, int) { return 100; }
    __host__ __device__ static int row_extent(const Args &, int64_t, int cols) { return cols; }
    // the row's mean and rstd, written by one thread per row when asked for
    __device__ __forceinline__ static void store_stats(const Args &a, int64_t row, float mean,
                                                       float rstd) {
        if (a.mean_out) a.mean_out[row] = mean;
        if (a.rstd_out) a.rstd_out[row] = rstd;
    }
};

// Row softmax: y = exp(x - max) / sum exp(x - max), the row held in
// registers (one HBM read, one write).  "PyTorch operator fusion in
// practice" (0539edu.com) §4.1-4.2 and "Operator fusion and kernel
// optimisation" (plumephp.com) §3.2: the softmax of a score row, normalised
// by the row maximum.  exp(d) = 2^(d log2 e) on the SFU.
template <typename TT> struct SoftmaxChain {
    using T = TT;
    static constexpr int kInputs = 1;
    static constexpr int kVec = Elem<T>::kVec;
    static constexpr bool kRegCap = false;     // see LnActChain
    static constexpr int kRowsTarget = 0;
    static constexpr int kWideScalarSlots = 32;   // see LnActChain
    static constexpr bool kShiftOk = true;        // see LnActChain
    // one input and no per-column vectors: 32 values per thread on the
    // cluster path (softmax fp32 at 40000 columns 4.5% faster than 16)
    static constexpr int kClusterVals = 32;
    // on the cluster path a CTA slice of 64 KB or more is staged: fp32 rows
    // through the ring into registers (131072 columns: 6.0 TB/s against 5.5
    // direct), bf16 rows held in the ring (rows_cluster_smem_kernel; 4.9
    // against 4.0)
    static constexpr bool kStageLargeSlices = true;
    static constexpr bool kPartialRows = false;   // every row read whole
    static constexpr bool kTwoPass = true;
    static constexpr bool kMaxFirst = true;
    static constexpr bool kStorePre = false;
    struct Args {
        const T *in[1];
        T *out;
    };
    template <int VEC> struct PrePC {};
    template <int VEC> struct PostPC {};
    static constexpr int kPostPC = 0;
    static constexpr int kColArrays = 0;      // no per-column values
    __host__ __device__ __forceinline__ static const T *col_array(const Args &, int) { return nullptr; }
    // no per-column arrays: the shifted kernel's staged form is the ring
    // alone, for bf16 rows (GB300, about 400 MB moved: 7-23% faster at 2051
    // to 32767 columns; fp32 rows were mixed, -10% to +6%)
    static constexpr bool kShiftStaged = sizeof(T) == 2;
    template <int VEC> using Early = NoEarly;
    template <int VEC, bool ANYOFF = false>
    __device__ __forceinline__ static void early(const Args &, int64_t, Early<VEC> &) {}
    template <int VEC, class LD = ColsGlobal<true>>
    __device__ __forceinline__ static void load_pre(const Args &, int, PrePC<VEC> &,
                                                    const LD & = LD{}) {}
    template <int VEC, class LD = ColsGlobal<true>>
    __device__ __forceinline__ static void load_post(const Args &, int, PostPC<VEC> &,
                                                     const LD & = LD{}) {}
    template <int VEC>
    __device__ __forceinline__ static void pre(const Frag<T, VEC> (&in)[1], const PrePC<VEC> &,
                                               const Args &, int64_t, int, float (&v)[VEC]) {
#pragma unroll
        for (int e = 0; e < VEC; ++e) v[e] = in[0].f[e];
    }
    template <int VEC>
    __device__ __forceinline__ static void store_pre(const float (&)[VEC], const Args &, int64_t) {}
    __device__ __forceinline__ static float stat1(float mx, int, const Args &) { return mx; }
    // v <- exp(v - max); the second pass sums these
    template <int VEC>
    __device__ __forceinline__ static float p2(float (&v)[VEC], float mx) {
        constexpr float kLog2e = 1.4426950408889634f;
        if constexpr (VEC == 1) {
            v[0] = ex2_approx((v[0] - mx) * kLog2e);
            return v[0];
        } else {
            float2 acc = splat2(0.0f);
#pragma unroll
            for (int e = 0; e < VEC; e += 2) {
                const float2 t = mul2(add2(make_float2(v[e], v[e + 1]), splat2(-mx)), splat2(kLog2e));
                const float2 x = make_float2(ex2_approx(t.x), ex2_approx(t.y));
                v[e] = x.x;
                v[e + 1] = x.y;
                acc = add2(acc, x);
            }
            return acc.x + acc.y;
        }
    }
    __device__ __forceinline__ static float stat2(float sum, int, const Args &) {
        return 1.0f / sum;
    }
    __device__ __forceinline__ static void store_stats(const Args &, int64_t, float, float) {}
    static int outputs(const Args &) { return 1; }
    static int read_percent(const Args &, int64_t, int) { return 100; }
    // leading elements of row `row` the chain reads (the staged engines copy no more)
    __host__ __device__ static int row_extent(const Args &, int64_t, int cols) { return cols; }
    template <int VEC>
    __device__ __forceinline__ static void post(const float (&v)[VEC], float, float inv,
                                                const PostPC<VEC> &, const Args &, int64_t,
                                                const Early<VEC> &, float (&o)[VEC]) {
        if constexpr (VEC == 1) {
            o[0] = v[0] * inv;
        } else {
#pragma unroll
            for (int e = 0; e < VEC; e += 2) {
                const float2 y = mul2(make_float2(v[e], v[e + 1]), splat2(inv));
                o[e] = y.x;
                o[e + 1] = y.y;
            }
        }
    }
};

// Softmax of attention-score rows ("PyTorch operator fusion in practice"
// (0539edu.com) §4.1-4.2): v = x * scale (one fp32 multiply, the caller's
// 1/sqrt(d)); with a causal mask, key j of row i takes no part when
// j > (i mod period) + offset, and its output is 0.  The masked tail of a row
// is never read: the staged engines copy only the row's first
// row_extent() elements.
template <typename TT> struct ScaleMaskSoftmaxChain {
    using T = TT;
    static constexpr int kInputs = 1;
    static constexpr int kVec = Elem<T>::kVec;
    static constexpr bool kRegCap = false;
    static constexpr int kRowsTarget = 0;
    static constexpr int kWideScalarSlots = 32;   // see LnActChain
    static constexpr bool kShiftOk = true;        // see LnActChain
    // one input and no per-column vectors: 32 values per thread on the
    // cluster path (softmax fp32 at 40000 columns 4.5% faster than 16)
    static constexpr int kClusterVals = 32;
    // on the cluster path a CTA slice of 64 KB or more is staged: fp32 rows
    // through the ring into registers (131072 columns: 6.0 TB/s against 5.5
    // direct), bf16 rows held in the ring (rows_cluster_smem_kernel; 4.9
    // against 4.0)
    static constexpr bool kStageLargeSlices = true;
    // rows may end early (row_extent): the direct paths skip the loads of
    // slots wholly past a row's unmasked prefix
    static constexpr bool kPartialRows = true;
    static constexpr bool kTwoPass = true;
    static constexpr bool kMaxFirst = true;
    static constexpr bool kStorePre = false;
    struct Args {
        const T *in[1];
        T *out;
        float scale;
        int causal;
        int64_t period;
        int64_t offset;    // at most cols (larger masks nothing more)
        uint64_t recip;    // (2^64 - 1) / period, for row mod period on the device
    };
    template <int VEC> struct PrePC {};
    template <int VEC> struct PostPC {};
    static constexpr int kPostPC = 0;
    static constexpr int kColArrays = 0;      // no per-column values
    __host__ __device__ __forceinline__ static const T *col_array(const Args &, int) { return nullptr; }
    // its rows' unmasked prefixes vary: no staged form on shifted rows
    static constexpr bool kShiftStaged = false;
    template <int VEC> using Early = NoEarly;
    template <int VEC, bool ANYOFF = false>
    __device__ __forceinline__ static void early(const Args &, int64_t, Early<VEC> &) {}
    template <int VEC, class LD = ColsGlobal<true>>
    __device__ __forceinline__ static void load_pre(const Args &, int, PrePC<VEC> &,
                                                    const LD & = LD{}) {}
    template <int VEC, class LD = ColsGlobal<true>>
    __device__ __forceinline__ static void load_post(const Args &, int, PostPC<VEC> &,
                                                     const LD & = LD{}) {}
    // row mod period: on the device a multiply-high by the reciprocal gives
    // the quotient or one less (the reciprocal is rounded down and the row is
    // below 2^63), so one conditional subtraction finishes it
    __host__ __device__ static int64_t query_of(const Args &a, int64_t row) {
#ifdef __CUDA_ARCH__
        const uint64_t q = __umul64hi((uint64_t)row, a.recip);
        uint64_t r = (uint64_t)row - q * (uint64_t)a.period;
        if (r >= (uint64_t)a.period) r -= (uint64_t)a.period;
        return (int64_t)r;
#else
        return row % a.period;
#endif
    }
    // elements [0, end) of row `row` are unmasked
    __host__ __device__ static int row_extent(const Args &a, int64_t row, int cols) {
        if (!a.causal) return cols;
        const int64_t last = query_of(a, row) + a.offset;
        return last + 1 < cols ? (int)(last + 1) : cols;
    }
    template <int VEC>
    __device__ __forceinline__ static void pre(const Frag<T, VEC> (&in)[1], const PrePC<VEC> &,
                                               const Args &a, int64_t row, int col,
                                               float (&v)[VEC]) {
        const int end = row_extent(a, row, 1 << 30);
#pragma unroll
        for (int e = 0; e < VEC; ++e)
            v[e] = col + e < end ? __fmul_rn(in[0].f[e], a.scale) : -INFINITY;
    }
    template <int VEC>
    __device__ __forceinline__ static void store_pre(const float (&)[VEC], const Args &, int64_t) {}
    __device__ __forceinline__ static float stat1(float mx, int, const Args &) { return mx; }
    template <int VEC>
    __device__ __forceinline__ static float p2(float (&v)[VEC], float mx) {
        return SoftmaxChain<T>::template p2<VEC>(v, mx);
    }
    __device__ __forceinline__ static float stat2(float sum, int, const Args &) {
        return 1.0f / sum;
    }
    __device__ __forceinline__ static void store_stats(const Args &, int64_t, float, float) {}
    static int outputs(const Args &) { return 1; }
    // The share of the row read on average (the staged engines copy the
    // unmasked prefix only): the mean of min(q + offset + 1, cols) over the
    // query positions q = row mod period that the rows take, as a percent of
    // cols.
    static int read_percent(const Args &a, int64_t rows, int cols) {
        if (!a.causal || cols <= 0) return 100;
        const int64_t P = rows < a.period ? (rows > 0 ? rows : 1) : a.period;
        int64_t k = (int64_t)cols - a.offset - 1;     // positions whose prefix is shorter
        if (k < 0) k = 0;
        if (k > P) k = P;
        const double read = (double)k * (double)(k - 1) / 2.0 + (double)k * (double)(a.offset + 1) +
                            (double)(P - k) * (double)cols;
        const int pct = (int)(100.0 * read / ((double)P * (double)cols) + 0.5);
        return pct < 1 ? 1 : (pct > 100 ? 100 : pct);
    }
    // y = e * (1 / sum); masked elements hold exp(-inf) = 0
    template <int VEC>
    __device__ __forceinline__ static void post(const float (&v)[VEC], float, float inv,
                                                const PostPC<VEC> &, const Args &, int64_t,
                                                const Early<VEC> &, float (&o)[VEC]) {
        if constexpr (VEC == 1) {
            o[0] = v[0] * inv;
        } else {
#pragma unroll
            for (int e = 0; e < VEC; e += 2) {
                const float2 y = mul2(make_float2(v[e], v[e + 1]), splat2(inv));
                o[e] = y.x;
                o[e + 1] = y.y;
            }
        }
    }
};

}  // namespace mb
