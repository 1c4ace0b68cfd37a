// chains.cuh -- the per-element arithmetic of the two reduce-plus-pointwise
// chains, plugged into the row engines of rows.cuh.
#pragma once

#include "rows.cuh"

namespace mb {

// Residual + LayerNorm + affine + GeLU-tanh.
// "Operator fusion and kernel optimisation" (plumephp.com) §2.2-2.3: v = x +
// residual, row mean and variance, rsqrt(var + eps), (v - mean) * inv_std *
// weight + bias, then GeLU (tanh form).  "Kernel fusion" course chapter 4
// (5688vip.com) §4.3: the variance as a second pass, sum((v - mean)^2) / cols.
template <typename TT> struct LnGeluChain {
    using T = TT;
    static constexpr int kInputs = 2;     // x, r
    static constexpr bool kTwoPass = true;
    static constexpr bool kMaxFirst = false;
    static constexpr bool kStorePre = false;
    struct Args {
        const T *in[2];
        const T *w;
        const T *b;
        T *out;
        float eps;
    };
    // per-column values of one slot: none before the reduction, w and b after
    template <int VEC> struct PrePC {};
    template <int VEC> struct PostPC { Frag<T, VEC> w, b; };
    static constexpr int kPostPC = 2;     // per-column vectors the epilogue reads
    template <int VEC>
    __device__ __forceinline__ static void load_pre(const Args &, int, PrePC<VEC> &) {}
    template <int VEC>
    __device__ __forceinline__ static void load_post(const Args &a, int col, PostPC<VEC> &pc) {
        pc.w.load_cached(a.w + col);
        pc.b.load_cached(a.b + col);
    }
    template <int VEC>
    __device__ __forceinline__ static void pre(const Frag<T, VEC> (&in)[2], const PrePC<VEC> &,
                                               const Args &, float (&v)[VEC]) {
#pragma unroll
        for (int e = 0; e < VEC; ++e) v[e] = __fadd_rn(in[0].f[e], in[1].f[e]);
    }
    // mean = sum(v) / H; second pass sum((v - mean)^2); rstd = 1/sqrt(var + eps)
    __device__ __forceinline__ static float stat1(float sum, int cols, const Args &) {
        return sum / (float)cols;
    }
    __device__ __forceinline__ static float p2(float &v, float mean, float acc) {
        const float d = v - mean;
        return fmaf(d, d, acc);
    }
    __device__ __forceinline__ static float stat2(float m2, int cols, const Args &a) {
        return rsqrtf(m2 / (float)cols + a.eps);
    }
    template <int VEC>
    __device__ __forceinline__ static void store_pre(const float (&)[VEC], const Args &, int64_t) {}
    template <int VEC>
    __device__ __forceinline__ static void post(const float (&v)[VEC], float mean, float rstd,
                                                const PostPC<VEC> &pc, const Args &,
                                                float (&o)[VEC]) {
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
            const float xhat = (v[e] - mean) * rstd;
            o[e] = gelu_tanh_f(fmaf(xhat, pc.w.f[e], pc.b.f[e]));
        }
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
    template <int VEC>
    __device__ __forceinline__ static void load_pre(const Args &a, int col, PrePC<VEC> &pc) {
        pc.bias.load_cached(a.bias + col);
    }
    template <int VEC>
    __device__ __forceinline__ static void load_post(const Args &a, int col, PostPC<VEC> &pc) {
        pc.gamma.load_cached(a.gamma + col);
        pc.beta.load_cached(a.beta + col);
    }
    template <int VEC>
    __device__ __forceinline__ static void pre(const Frag<T, VEC> (&in)[1],
                                               const PrePC<VEC> &pc, const Args &a,
                                               float (&v)[VEC]) {
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
            const float t = __fadd_rn(__fmul_rn(in[0].f[e], a.x_scale), pc.bias.f[e]);
            const float r = relu_f(t);
            const float p = __fmul_rn(r, r);
            const float q = __fmul_rn(r, a.branch_scale);
            v[e] = __fadd_rn(p, q);
        }
    }
    // m = sum(s) / cols (a row sum divided by the row length); no second pass
    __device__ __forceinline__ static float stat1(float sum, int cols, const Args &) {
        return sum / (float)cols;
    }
    __device__ __forceinline__ static float p2(float &, float, float acc) { return acc; }
    __device__ __forceinline__ static float stat2(float, int, const Args &) { return 0.0f; }
    template <int VEC>
    __device__ __forceinline__ static void store_pre(const float (&)[VEC], const Args &, int64_t) {}
    template <int VEC>
    __device__ __forceinline__ static void post(const float (&v)[VEC], float mean, float,
                                                const PostPC<VEC> &pc, const Args &,
                                                float (&o)[VEC]) {
#pragma unroll
        for (int e = 0; e < VEC; ++e)
            o[e] = __fadd_rn(__fmul_rn(__fsub_rn(v[e], mean), pc.gamma.f[e]), pc.beta.f[e]);
    }
};
using InductorChain = InductorChainT<float>;

// LayerNorm family: v = x (+ r); optionally h = v written out (the residual
// stream); out = act((v - mean) * rstd * w + b), act none / relu / gelu-tanh.
// "Kernel fusion" course chapter 4 (5688vip.com) §4.3 (LayerNorm, two-pass
// variance); "Operator fusion and kernel optimisation" (plumephp.com) §2.1
// (LayerNorm -> ReLU in one kernel) and §2.2-2.3 (residual + LayerNorm + GeLU).
enum { kActNone = 0, kActRelu = 1, kActGelu = 2 };
template <typename TT, bool RES> struct LnActChain {
    using T = TT;
    static constexpr int kInputs = RES ? 2 : 1;
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
    };
    template <int VEC> struct PrePC {};
    template <int VEC> struct PostPC { Frag<T, VEC> w, b; };
    static constexpr int kPostPC = 2;
    template <int VEC>
    __device__ __forceinline__ static void load_pre(const Args &, int, PrePC<VEC> &) {}
    template <int VEC>
    __device__ __forceinline__ static void load_post(const Args &a, int col, PostPC<VEC> &pc) {
        pc.w.load_cached(a.w + col);
        pc.b.load_cached(a.b + col);
    }
    template <int VEC>
    __device__ __forceinline__ static void pre(const Frag<T, VEC> (&in)[kInputs],
                                               const PrePC<VEC> &, const Args &,
                                               float (&v)[VEC]) {
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
            if constexpr (RES) v[e] = __fadd_rn(in[0].f[e], in[1].f[e]);
            else v[e] = in[0].f[e];
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
    __device__ __forceinline__ static float stat1(float sum, int cols, const Args &) {
        return sum / (float)cols;
    }
    __device__ __forceinline__ static float p2(float &v, float mean, float acc) {
        const float d = v - mean;
        return fmaf(d, d, acc);
    }
    __device__ __forceinline__ static float stat2(float m2, int cols, const Args &a) {
        return rsqrtf(m2 / (float)cols + a.eps);
    }
    template <int VEC>
    __device__ __forceinline__ static void post(const float (&v)[VEC], float mean, float rstd,
                                                const PostPC<VEC> &pc, const Args &a,
                                                float (&o)[VEC]) {
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
            const float n = fmaf((v[e] - mean) * rstd, pc.w.f[e], pc.b.f[e]);
            o[e] = a.act == kActGelu ? gelu_tanh_f(n) : (a.act == kActRelu ? relu_f(n) : n);
        }
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
    template <int VEC>
    __device__ __forceinline__ static void load_pre(const Args &, int, PrePC<VEC> &) {}
    template <int VEC>
    __device__ __forceinline__ static void load_post(const Args &, int, PostPC<VEC> &) {}
    template <int VEC>
    __device__ __forceinline__ static void pre(const Frag<T, VEC> (&in)[1], const PrePC<VEC> &,
                                               const Args &, float (&v)[VEC]) {
#pragma unroll
        for (int e = 0; e < VEC; ++e) v[e] = in[0].f[e];
    }
    template <int VEC>
    __device__ __forceinline__ static void store_pre(const float (&)[VEC], const Args &, int64_t) {}
    __device__ __forceinline__ static float stat1(float mx, int, const Args &) { return mx; }
    // v <- exp(v - max); the second pass sums these
    __device__ __forceinline__ static float p2(float &v, float mx, float acc) {
        constexpr float kLog2e = 1.4426950408889634f;
        v = ex2_approx((v - mx) * kLog2e);
        return acc + v;
    }
    __device__ __forceinline__ static float stat2(float sum, int, const Args &) {
        return 1.0f / sum;
    }
    template <int VEC>
    __device__ __forceinline__ static void post(const float (&v)[VEC], float, float inv,
                                                const PostPC<VEC> &, const Args &,
                                                float (&o)[VEC]) {
#pragma unroll
        for (int e = 0; e < VEC; ++e) o[e] = v[e] * inv;
    }
};

}  // namespace mb
