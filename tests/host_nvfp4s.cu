// host_nvfp4s.cu -- the paired 4:8 sparse NVFP4 chunk decoding of the decode
// kernels (top_moe_expert_gb300/csrc/nvfp4s.cuh), run on the CPU for the CPU
// tests: each row's dot product with x is formed chunk by chunk through the
// kernels' own chunk function, with the chunk's bytes read at the offsets the
// kernels use (16c, 4c, 2c).
#include <cstdint>
#include <cstring>
#include "nvfp4s.cuh"

extern "C" void nv4_rows_dot(const uint8_t *v, const uint8_t *m, const uint8_t *s, float alpha, int rows, int K,
                             const float *x, double *out)
{
    for (int r = 0; r < rows; ++r) {
        double acc = 0.0;
        for (int c = 0; c < K / 64; ++c) {
            uint32_t w[4], meta;
            uint16_t sc2;
            std::memcpy(w, v + static_cast<int64_t>(r) * (K / 4) + 16 * c, 16);
            std::memcpy(&meta, m + static_cast<int64_t>(r) * (K / 16) + 4 * c, 4);
            std::memcpy(&sc2, s + static_cast<int64_t>(r) * (K / 32) + 2 * c, 2);
            acc += moe::nv4::chunk_dot(w, meta, sc2, x + 64 * c);
        }
        out[r] = acc * alpha;
    }
}
