// host_split.cu -- the single-token kernels' CTA split (pipe::cta_split in
// top_moe_expert_gb300/csrc/pipe_common.cuh, 32-bit arithmetic), run on the
// CPU for the CPU tests: every CTA's range of (route, neuron) pairs and of
// output rows, for one (nv, I, d, G) and a stage size of 4 or 8 neurons.
#include <cstdint>
#include "pipe_common.cuh"

extern "C" void split_all(int nv, int I, int d, int G, int RPS, int PS, int32_t *out)
{
    for (int c = 0; c < G; ++c) {
        const moe::pipe::Split s = PS == 4 ? moe::pipe::cta_split<4>(nv, I, d, c, G, RPS)
                                           : moe::pipe::cta_split<8>(nv, I, d, c, G, RPS);
        int32_t *o = out + 6 * c;
        o[0] = s.q_lo;
        o[1] = s.P;
        o[2] = s.S;
        o[3] = s.o0;
        o[4] = s.nrows;
        o[5] = s.SW;
    }
}
