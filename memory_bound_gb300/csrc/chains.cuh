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
    struct Args {
        const T *in[2];
        const T *w;
        const T *b;
        T *out;
        float eps;
    };
    template <int VEC>
    __device__ __forceinline__ static void pre(const Frag<T, VEC> (&in)[2], const Args &, int,
                                               float (&v)[VEC]) {
#pragma unroll
        for (int e = 0; e < VEC; ++e) v[e] = __fadd_rn(in[0].f[e], in[1].f[e]);
    }
    __device__ __forceinline__ static float rstd(float m2, int cols, const Args &a) {
        return rsqrtf(m2 / (float)cols + a.eps);
    }
    template <int VEC>
    __device__ __forceinline__ static void post(const float (&v)[VEC], float mean, float rstd,
                                                const Args &a, int col, float (&o)[VEC]) {
        Frag<T, VEC> w, b;
        w.load_cached(a.w + col);
        b.load_cached(a.b + col);
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
            const float xhat = (v[e] - mean) * rstd;
            o[e] = gelu_tanh_f(fmaf(xhat, w.f[e], b.f[e]));
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
    struct Args {
        const float *in[1];
        const float *bias;
        const float *gamma;
        const float *beta;
        float *out;
        float x_scale;
        float branch_scale;
    };
    template <int VEC>
    __device__ __forceinline__ static void pre(const Frag<float, VEC> (&in)[1], const Args &a,
                                               int col, float (&v)[VEC]) {
        Frag<float, VEC> bias;
        bias.load_cached(a.bias + col);
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
            const float t = __fadd_rn(__fmul_rn(in[0].f[e], a.x_scale), bias.f[e]);
            const float r = relu_f(t);
            const float p = __fmul_rn(r, r);
            const float q = __fmul_rn(r, a.branch_scale);
            v[e] = __fadd_rn(p, q);
        }
    }
    __device__ __forceinline__ static float rstd(float, int, const Args &) { return 0.0f; }
    template <int VEC>
    __device__ __forceinline__ static void post(const float (&v)[VEC], float mean, float,
                                                const Args &a, int col, float (&o)[VEC]) {
        Frag<float, VEC> g, b;
        g.load_cached(a.gamma + col);
        b.load_cached(a.beta + col);
#pragma unroll
        for (int e = 0; e < VEC; ++e)
            o[e] = __fadd_rn(__fmul_rn(__fsub_rn(v[e], mean), g.f[e]), b.f[e]);
    }
};

}  // namespace mb
