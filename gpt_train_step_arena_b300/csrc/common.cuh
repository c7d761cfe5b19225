// Shared device helpers for the GPT-2 train-step kernels (sm_103a).
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

typedef __nv_bfloat16 bf16;

#define G2_DEV __device__ __forceinline__

#include <utility>

namespace g2 {
void count_launches(unsigned n);
// Programmatic stream serialization: off by default, on with the environment variable
// G2_PDL=1 (read once).  Results are identical either way.  On a power-capped B300 it
// removes launch gaps but raises the average power, and the lower clock that follows
// cost more than the gaps (124M step: 33.2 ms with it, 32.9 ms without).
bool pdl_enabled();
// Every kernel of the library is launched through this: counts the launch and launches it,
// with programmatic stream serialization when enabled (the next kernel on the stream is
// then scheduled while the current one drains).  Every kernel begins with G2_PDL_ENTRY(),
// which waits until the preceding kernel has completed (and its memory is visible) before
// touching global memory, so the order of the stream is the same either way.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_k(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                            Args&&... args) {
    count_launches(1);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = pdl_enabled() ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}
// The same for a kernel launched in clusters of `cluster_x` consecutive CTAs.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_k_cluster(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                                    unsigned cluster_x, Args&&... args) {
    count_launches(1);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute at[2];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = cluster_x;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = pdl_enabled() ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}
}  // namespace g2
// First statement of every kernel: wait for the kernel before it on the stream (all of
// its work done and visible), then let the next one be scheduled.
#define G2_PDL_ENTRY()                                                   \
    do {                                                                 \
        asm volatile("griddepcontrol.wait;" ::: "memory");               \
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");  \
    } while (0)

G2_DEV float to_f(float x) { return x; }
G2_DEV float to_f(bf16 x) { return __bfloat162float(x); }

template <typename T> G2_DEV T from_f(float x);
template <> G2_DEV float from_f<float>(float x) { return x; }
template <> G2_DEV bf16 from_f<bf16>(float x) { return __float2bfloat16_rn(x); }

G2_DEV float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
G2_DEV float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// 8 consecutive elements moved as one 16-byte (bf16) or two 16-byte (fp32) accesses.
template <typename T> struct Vec8;
template <> struct Vec8<bf16> {
    static G2_DEV void load(const bf16* p, float* f) {
        uint4 u = *reinterpret_cast<const uint4*>(p);
        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
        for (int i = 0; i < 4; i++) {
            float2 t = __bfloat1622float2(h[i]);
            f[2 * i] = t.x;
            f[2 * i + 1] = t.y;
        }
    }
    static G2_DEV void store(bf16* p, const float* f) {
        uint4 u;
        __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
        for (int i = 0; i < 4; i++) h[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
        *reinterpret_cast<uint4*>(p) = u;
    }
};
template <> struct Vec8<float> {
    static G2_DEV void load(const float* p, float* f) {
        float4 a = *reinterpret_cast<const float4*>(p);
        float4 b = *reinterpret_cast<const float4*>(p + 4);
        f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
        f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
    }
    static G2_DEV void store(float* p, const float* f) {
        *reinterpret_cast<float4*>(p) = make_float4(f[0], f[1], f[2], f[3]);
        *reinterpret_cast<float4*>(p + 4) = make_float4(f[4], f[5], f[6], f[7]);
    }
};

// GELU, tanh form (llm.c annotated listing §1.9; picoGPT gelu).
G2_DEV float gelu_tanh(float x) {
    const float k = 0.7978845608028654f;  // sqrt(2/pi)
    float u = k * (x + 0.044715f * x * x * x);
    return 0.5f * x * (1.0f + tanhf(u));
}
// Its derivative (llm.c §1.10) with sech^2(u) written as 1 - tanh^2(u).
G2_DEV float gelu_tanh_grad(float x) {
    const float k = 0.7978845608028654f;
    float u = k * (x + 0.044715f * x * x * x);
    float th = tanhf(u);
    float sech2 = 1.0f - th * th;
    return 0.5f * (1.0f + th) + x * 0.5f * sech2 * k * (1.0f + 3.0f * 0.044715f * x * x);
}

// tanh through the identity tanh(u) = 1 - 2 / (e^{2u} + 1), with the hardware base-2
// exponential and reciprocal approximations: absolute error a few 1e-7, far below a bf16
// rounding; used where the result is rounded to bf16 (the tensor-core GEMM epilogues).
// Saturates correctly: e^{2u} -> inf gives 1, e^{2u} -> 0 gives -1.
G2_DEV float tanh_via_exp2(float u) {
    float e, r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(u * 2.8853900817779268f));  // 2 log2(e) u
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(e + 1.0f));
    return fmaf(-2.0f, r, 1.0f);
}
G2_DEV float gelu_tanh_fast(float x) {
    const float k = 0.7978845608028654f;
    float u = k * (x + 0.044715f * x * x * x);
    return 0.5f * x * (1.0f + tanh_via_exp2(u));
}
G2_DEV float gelu_tanh_grad_fast(float x) {
    const float k = 0.7978845608028654f;
    float u = k * (x + 0.044715f * x * x * x);
    float th = tanh_via_exp2(u);
    float sech2 = 1.0f - th * th;
    return 0.5f * (1.0f + th) + x * 0.5f * sech2 * k * (1.0f + 3.0f * 0.044715f * x * x);
}

// Instruction-count helpers for the element-wise passes that are bound by issue slots:
// the hardware 2^x (relative error about 2^-22, results below 2^-126 flush to zero), a
// three-input maximum, and two-wide fp32 arithmetic (each lane rounded once, exactly as
// the scalar fmaf / +).
G2_DEV float ex2_ftz(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
G2_DEV float max3f(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}
G2_DEV float2 fma2(float2 a, float2 b, float2 c) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
        "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}
G2_DEV float2 add2(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}
G2_DEV float2 sub2(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "sub.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}
G2_DEV float2 mul2(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}
// GELU (tanh form) and its derivative on two values, for the GEMM epilogues.  With
// r = 1 / (e + 1), e = 2^(2 log2(e) u) = e^{2u}, tanh(u) = 1 - 2r, so
//   gelu(x)  = 0.5 x (1 + tanh u)                      = x (1 - r)
//   gelu'(x) = 0.5 (1 + tanh u) + 0.5 x sech^2(u) u'   = (1 - r) (1 + 2 k x r (1 + 3 c x^2))
// with u = k (x + c x^3), k = sqrt(2/pi), c = 0.044715 and sech^2 = 1 - tanh^2 = 4 r (1 - r):
// the same exponential and reciprocal approximations as the scalar forms, in about half
// the instructions (results differ from them by a few rounding steps, far below a bf16
// rounding).  Saturation: e -> inf gives r = 0 (gelu = x, gelu' = 1); e -> 0 gives r = 1
// (gelu = 0, gelu' = 0).
G2_DEV float rcp_approx(float x) {
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}
G2_DEV float2 gelu_r2(float2 x, float2& r) {  // r of both values (returned through r), x^2
    constexpr float K2 = 2.0f * 1.4426950408889634f * 0.7978845608028654f;  // 2 log2(e) k
    constexpr float C2 = K2 * 0.044715f;
    const float2 x2 = mul2(x, x);
    const float2 u = mul2(x, fma2(x2, make_float2(C2, C2), make_float2(K2, K2)));
    r = make_float2(rcp_approx(ex2_ftz(u.x) + 1.0f), rcp_approx(ex2_ftz(u.y) + 1.0f));
    return x2;
}
G2_DEV float2 gelu2(float2 x) {
    float2 r;
    gelu_r2(x, r);
    return fma2(make_float2(-x.x, -x.y), r, x);  // x - x r
}
G2_DEV float2 gelu_grad2(float2 x) {
    constexpr float K = 0.7978845608028654f, C = 0.044715f;
    float2 r;
    const float2 x2 = gelu_r2(x, r);
    const float2 a = fma2(r, make_float2(-1.f, -1.f), make_float2(1.f, 1.f));                    // 1 - r
    const float2 poly = fma2(x2, make_float2(6.f * K * C, 6.f * K * C), make_float2(2.f * K, 2.f * K));  // 2k (1 + 3c x^2)
    const float2 b = fma2(mul2(x, r), poly, make_float2(1.f, 1.f));
    return mul2(a, b);
}
// the two bf16 halves of a 32-bit word as fp32 (exact)
G2_DEV float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
G2_DEV float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
// (lo, hi) rounded to nearest-even bf16 and packed into one word, lo in the low half
G2_DEV uint32_t pack_bf16x2_rn(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
}

// Device-side error flags (bitwise OR into one int): never trap, the host reads them.
enum {
    G2_FLAG_BAD_TOKEN = 1,
    G2_FLAG_BAD_TARGET = 2,
    G2_FLAG_NONFINITE = 4,
    G2_FLAG_TIMEOUT = 8,
};
