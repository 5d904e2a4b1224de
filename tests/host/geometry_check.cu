// Host-side check of two invariants the step kernel relies on (compiled and
// run by tests/test_host_geometry.py; nothing here runs on a GPU):
//  - every stage geometry the weight stream can use has a power-of-two row
//    count and segments-per-row count (the kernels shift instead of divide);
//  - it / ns == umulhi(it, ring_magic(ns)) for every ring depth (at least
//    two slots, as the set-up enforces) and every stage counter a launch can
//    reach.
#include <cstdint>
#include <cstdio>

#include "kernels.h"
#include "gemv_core.cuh"

int main() {
    using namespace tts;
    int checked = 0, not_pow2 = 0;
    for (int prec = 0; prec < 2; ++prec)
        for (int epi = 0; epi < 3; ++epi)
            for (int K = 128; K <= 16384; K += 128) {
                const StageGeom g = stage_geom(prec, epi, K);
                if (!g.ok) continue;
                ++checked;
                if ((g.rs & (g.rs - 1)) || (g.wpr & (g.wpr - 1)) || g.rs < 1 || g.wpr < 1) ++not_pow2;
            }
    long long wrong = 0, pairs = 0;
    for (int ns = 2; ns <= 32; ++ns) {
        const uint32_t m = core::ring_magic(ns);
        for (uint32_t it = 0; it < (1u << 22); ++it, ++pairs)
            if ((uint32_t)(((uint64_t)it * m) >> 32) != it / (uint32_t)ns) ++wrong;
    }
    std::printf("geometries %d not_pow2 %d pairs %lld wrong %lld\n", checked, not_pow2, pairs, wrong);
    return (checked > 0 && not_pow2 == 0 && wrong == 0) ? 0 : 1;
}
