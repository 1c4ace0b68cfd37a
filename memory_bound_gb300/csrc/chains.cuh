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
// the row sum never leaves the chip (§08 of the same post).
struct InductorChain {
    using T = float;
    static constexpr int kInputs = 1;     // x
    static constexpr bool kTwoPass = false;
    static constexpr bool kMaxFirst = false;
    struct Args {
        const float *in[1];
        const float *bias;
        const float *gamma;
        const float *beta;
        float *out;
        float x_scale;
        float branch_scale;
    };
    // per-column values of one slot: bias before the reduction, gamma and beta after
    template <int VEC> struct PrePC { Frag<float, VEC> bias; };
    template <int VEC> struct PostPC { Frag<float, VEC> gamma, beta; };
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
    __device__ __forceinline__ static void pre(const Frag<float, VEC> (&in)[1],
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
    __device__ __forceinline__ static void post(const float (&v)[VEC], float mean, float,
                                                const PostPC<VEC> &pc, const Args &,
                                                float (&o)[VEC]) {
#pragma unroll
        for (int e = 0; e < VEC; ++e)
            o[e] = __fadd_rn(__fmul_rn(__fsub_rn(v[e], mean), pc.gamma.f[e]), pc.beta.f[e]);
    }
};

}  // namespace mb
