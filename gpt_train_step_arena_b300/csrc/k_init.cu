// Seeded initial parameters on the device (gpt2_init_params).
//
// The generator is xorshift64* (llm.c annotated listing §1.33 random_u32) with the float
// mapping of §1.34 random_f32 (top 24 bits / 2^24), run as LANES independent streams:
// lane j starts from splitmix64(seed + j) (never 0), and draw i of a request comes from
// lane i % LANES in round i / LANES; every request uses whole rounds (draws past its end
// are discarded).  Normal values come in Box-Muller pairs from consecutive draws (u1, u2)
// with u1 kept at or above 1e-7: z0 = r cos(2 pi u2), z1 = r sin(2 pi u2), r =
// sqrt(-2 ln u1), computed in double and rounded to float once after scaling by the
// standard deviation.  The rule: every weight matrix, wte and wpe ~ N(0, 0.02), the two
// residual projections ~ N(0, 0.02 / sqrt(2 L)), biases 0, LayerNorm gains 1, shifts 0,
// padded vocabulary rows 0; tensors draw in the listing's parameter order (§1.16).
#include <cmath>

#include "common.cuh"
#include "kernels.h"

namespace g2 {

namespace {

constexpr int LANES = 1 << 16;
constexpr int PAIRS = LANES / 2;  // one thread per lane pair (2p, 2p+1)

G2_DEV uint64_t splitmix64(uint64_t x) {
    uint64_t z = x + 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    z = z ^ (z >> 31);
    return z ? z : 0x9E3779B97F4A7C15ull;
}

G2_DEV uint32_t xorshift64star(uint64_t& s) {
    s ^= s >> 12;
    s ^= s << 25;
    s ^= s >> 27;
    return (uint32_t)((s * 0x2545F4914F6CDD1Dull) >> 32);
}

// (u32 >> 8) / 2^24: exact in float and in double
G2_DEV double unit(uint32_t u) { return (double)(u >> 8) * (1.0 / 16777216.0); }

// Thread p owns lanes 2p and 2p+1: the two draws of pair j = round * PAIRS + p of every
// normal tensor, so its outputs 2j, 2j+1 sit next to those of threads p-1 and p+1.
__global__ void __launch_bounds__(256) init_normal_k(float* params, InitPlan plan, uint64_t seed) {
    G2_PDL_ENTRY();
    const int p = blockIdx.x * blockDim.x + threadIdx.x;
    if (p >= PAIRS) return;
    uint64_t s0 = splitmix64(seed + 2ull * p), s1 = splitmix64(seed + 2ull * p + 1);
    const double two_pi = 6.283185307179586;  // 2 * pi rounded to double
    for (int k = 0; k < plan.count; k++) {
        float* out = params + plan.offset[k];
        const size_t n = plan.n[k];
        const double std = plan.std[k];
        const size_t rounds = (2 * ((n + 1) / 2) + LANES - 1) / LANES;
        for (size_t r = 0; r < rounds; r++) {
            const uint32_t a = xorshift64star(s0), b = xorshift64star(s1);
            const size_t j = r * PAIRS + p;
            if (2 * j >= n) continue;  // past the end: the draw is discarded
            const double u1 = fmax(unit(a), 1e-7), u2 = unit(b);
            const double rad = sqrt(-2.0 * log(u1));
            const double ang = two_pi * u2;
            out[2 * j] = __double2float_rn(rad * cos(ang) * std);
            if (2 * j + 1 < n) out[2 * j + 1] = __double2float_rn(rad * sin(ang) * std);
        }
    }
}

__global__ void fill_k(float* p, size_t n, float v) {
    G2_PDL_ENTRY();
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
        p[i] = v;
}

}  // namespace

cudaError_t init_params_device(float* params, const InitPlan& plan, const float* const* ones, const size_t* ones_n,
                               int n_ones, uint64_t seed, cudaStream_t s) {
    for (int i = 0; i < n_ones; i++) {
        if (!ones_n[i]) continue;
        const unsigned blocks = (unsigned)std::min<size_t>((ones_n[i] + 255) / 256, 1024);
        ::g2::launch_k(fill_k, blocks, 256, 0, s, const_cast<float*>(ones[i]), ones_n[i], 1.0f);
    }
    ::g2::launch_k(init_normal_k, PAIRS / 256, 256, 0, s, params, plan, seed);
    return cudaGetLastError();
}

}  // namespace g2
