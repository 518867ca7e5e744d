// launch_staged.cuh -- picks the staged_kernel instance for a plan.
#pragma once

#include <type_traits>

#include "launch_util.h"
#include "planner.h"
#include "staged.cuh"

namespace rmsn {

template <typename T, int MODE, int NT, int G, int V, bool GEN, bool SH, bool CLAIM = false>
cudaError_t launch_staged_inst(const Plan &p, const KernelArgs &a, cudaStream_t stream) {
    constexpr int MINB = staged_max_ctas_per_sm(MODE, NT, G, V);
    static std::atomic<uint64_t> smem_mask{0};
    auto kern = staged_kernel<T, MODE, NT, G, V, MINB, GEN, SH, CLAIM>;
    cudaError_t e = allow_max_dynamic_smem((const void *)kern, smem_mask);
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, dim3(p.grid), dim3(NT), p.smem, stream, a);
}

// Column boxes for the tensor maps: the fewest boxes of equal width that
// tile D, at most 2 KB wide (256 units of 8 bytes, the TMA box limit) and a
// multiple of 16 bytes; 0 if four boxes do not do it.  Rows of the sub-warp
// shape (at most 2 KB) take one box.
inline int tmap_boxes(int64_t D, int es) {
    for (int n = 1; n <= 4; ++n)
        if (D % n == 0 && D / n * es <= 2048 && (D / n * es) % 16 == 0) return n;
    return 0;
}

// The dense instance unless a tensor the mode uses has rows a stride apart
// or rstd is given.  General sub-warp tiles go through 2-D tensor maps when
// D splits into boxes (one copy per box instead of one per row), else one
// bulk copy per row.  SH: the shifted-rows instances (dense rows whose
// tensors share one offset from a 16-byte boundary; the plan says so).
template <typename T, int MODE, int NT, int G, int V>
cudaError_t launch_staged_general(const Plan &p, const KernelArgs &a, cudaStream_t stream) {
    const int64_t D = a.D;
    bool gen = a.rstd != nullptr || a.ld_in0 != D || a.ld_out0 != D;
    if constexpr (input_tensors(MODE) >= 2) gen = gen || a.ld_in1 != D;
    if constexpr (input_tensors(MODE) == 3) gen = gen || a.ld_in2 != D;
    if constexpr (MODE == MODE_FWD_RES) gen = gen || a.ld_out1 != D;
    // The dense CTA-per-row forwards of at least CLAIM_MIN_NT threads have a
    // claimed-tiles instance, launched when the call hands them counters.
    if constexpr (!is_vjp(MODE) && G == NT && NT >= CLAIM_MIN_NT)
        if (!gen && a.tile_ctr)
            return launch_staged_inst<T, MODE, NT, G, V, false, false, true>(p, a, stream);
    if (!gen) return launch_staged_inst<T, MODE, NT, G, V, false, false>(p, a, stream);
    if constexpr (G == NT) {
        return launch_staged_inst<T, MODE, NT, G, V, true, false>(p, a, stream);
    } else {
        constexpr int es = (int)sizeof(T);
        constexpr int dtype = es == 4 ? 2 : std::is_same<T, __half>::value ? 0 : 1;
        KernelArgs b = a;
        b.box_cols = a.D;
        b.use_tmap = 0;
        const int n = tmap_boxes(D, es);
        const int64_t box_bytes = n ? (int64_t)p.tile_rows * (D / n) * es : 0;
        // every box lands 128-byte aligned; row coordinates fit in int32
        if (n && box_bytes % 128 == 0 && p.tile_rows <= 256 && a.rows <= INT32_MAX &&
            planner::tuning().tmap) {
            const void *ins[3] = {a.in0, a.in1, a.in2};
            const int64_t lds[3] = {a.ld_in0, a.ld_in1, a.ld_in2};
            bool ok = true;
            for (int i = 0; i < input_tensors(MODE) && ok; ++i)
                ok = encode_rows_tmap(&b.tmap[i], ins[i], a.rows, D, lds[i], dtype,
                                      (int)(D / n), p.tile_rows);
            if (ok) {
                b.box_cols = (int)(D / n);
                b.use_tmap = 1;
            }
        }
        return launch_staged_inst<T, MODE, NT, G, V, true, false>(p, b, stream);
    }
}

template <typename T, int MODE, int NT, int G, int V, bool SH>
cudaError_t launch_staged_one(const Plan &p, const KernelArgs &a, cudaStream_t stream) {
    if constexpr (SH)
        return launch_staged_inst<T, MODE, NT, G, V, false, true>(p, a, stream);
    else
        return launch_staged_general<T, MODE, NT, G, V>(p, a, stream);
}

template <typename T, int MODE, bool SH>
cudaError_t launch_staged_mode(const Plan &p, const KernelArgs &a, cudaStream_t s) {
    static_assert(N_STAGED_CFG == 19, "keep this switch in step with STAGED_CFGS");
    switch (p.cfg) {
        case 0: return launch_staged_one<T, MODE, 256, 8, 1, SH>(p, a, s);
        case 1: return launch_staged_one<T, MODE, 256, 16, 1, SH>(p, a, s);
        case 2: return launch_staged_one<T, MODE, 256, 32, 1, SH>(p, a, s);
        case 3: return launch_staged_one<T, MODE, 256, 32, 2, SH>(p, a, s);
        case 4: return launch_staged_one<T, MODE, 256, 32, 3, SH>(p, a, s);
        case 5: return launch_staged_one<T, MODE, 256, 32, 4, SH>(p, a, s);
        case 6: return launch_staged_one<T, MODE, 128, 128, 2, SH>(p, a, s);
        case 7: return launch_staged_one<T, MODE, 256, 256, 2, SH>(p, a, s);
        case 8: return launch_staged_one<T, MODE, 512, 512, 2, SH>(p, a, s);
        case 9: return launch_staged_one<T, MODE, 1024, 1024, 2, SH>(p, a, s);
        case 10:
            if constexpr (is_vjp(MODE)) return cudaErrorInvalidValue;
            else return launch_staged_one<T, MODE, 256, 256, 4, SH>(p, a, s);
        case 11: return launch_staged_one<T, MODE, 96, 96, 2, SH>(p, a, s);
        case 12: return launch_staged_one<T, MODE, 192, 192, 2, SH>(p, a, s);
        case 13: return launch_staged_one<T, MODE, 384, 384, 2, SH>(p, a, s);
        case 14: return launch_staged_one<T, MODE, 768, 768, 2, SH>(p, a, s);
        case 15: return launch_staged_one<T, MODE, 160, 160, 2, SH>(p, a, s);
        case 16: return launch_staged_one<T, MODE, 224, 224, 2, SH>(p, a, s);
        case 17: return launch_staged_one<T, MODE, 320, 320, 2, SH>(p, a, s);
        case 18: return launch_staged_one<T, MODE, 448, 448, 2, SH>(p, a, s);
        default: return cudaErrorInvalidValue;
    }
}

template <typename T, bool SH>
cudaError_t launch_staged_t(int mode, const Plan &p, const KernelArgs &a, cudaStream_t s) {
    switch (mode) {
        case MODE_FWD_RES: return launch_staged_mode<T, MODE_FWD_RES, SH>(p, a, s);
        case MODE_FWD_NORES: return launch_staged_mode<T, MODE_FWD_NORES, SH>(p, a, s);
        case MODE_VJP: return launch_staged_mode<T, MODE_VJP, SH>(p, a, s);
        case MODE_VJP_ADD: return launch_staged_mode<T, MODE_VJP_ADD, SH>(p, a, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace rmsn
