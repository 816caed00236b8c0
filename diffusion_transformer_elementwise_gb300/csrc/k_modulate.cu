// k_modulate.cu -- out = rms_norm(x, eps) * (1 + scale) + shift on GB300.
//
// Operation: prhub summary of sglang PR #34172 (LTX-2 quality=high fused
// RMSNorm+modulate), section "key source snippet" (the expression of
// _ltx2_rms_norm_modulate) and section "implementation breakdown", item 2
// (weightless RMSNormNoWeight, the whole expression in one launch).
//
// 16-byte aligned rows of up to 8 KB: two warps per row (dit_wrow.cuh);
// other 16-byte aligned rows, the E4M3 output and the grouped launch: the
// staged CTA-per-row kernel (dit_pipe.cuh); unaligned rows: the phased staged
// kernel or the register kernel; long rows: the two-pass kernel
// (dit_rows.cuh).
#include "dit_rows.cuh"

namespace dit {

cudaError_t launch_modulate(const DeviceInfo& dev, int dtype, int vb, bool mod_full,
                            const RowArgs& a, int64_t B, cudaStream_t stream) {
  return mod_full ? launch_row_op<OP_MOD, false, true>(dev, dtype, vb, a, B, stream)
                  : launch_row_op<OP_MOD, false, false>(dev, dtype, vb, a, B, stream);
}

cudaError_t launch_modulate_fp8(const DeviceInfo& dev, int dtype, bool mod_full,
                                const RowArgs& a, int64_t B, cudaStream_t stream) {
  return with_statistic<OP_MOD>(a.exact, [&](auto ex) {
    constexpr bool EX = decltype(ex)::value;
    if constexpr (EX) {
      // the exact statistic: two warps per row (the staged kernel's exact
      // instantiation for E4M3 spills; on [1,32640,4096] bf16 it took 194 us)
      const cudaError_t w =
          mod_full ? launch_wrow<OP_MOD, false, true, true, true>(dev, dtype, a, B, stream)
                   : launch_wrow<OP_MOD, false, false, true, true>(dev, dtype, a, B, stream);
      if (w != cudaErrorNotSupported) return w;
    }
    return mod_full ? launch_pipe<OP_MOD, false, true, true, EX>(dev, dtype, a, B, stream)
                    : launch_pipe<OP_MOD, false, false, true, EX>(dev, dtype, a, B, stream);
  });
}

cudaError_t launch_modulate_grouped(const DeviceInfo& dev, int dtype, bool mod_full,
                                    const RowArgs* a, const int64_t* B, int count,
                                    cudaStream_t stream) {
  return with_statistic<OP_MOD>(count > 0 && a[0].exact, [&](auto ex) {
    constexpr bool EX = decltype(ex)::value;
    return mod_full ? launch_pipe_grouped<OP_MOD, false, true, EX>(dev, dtype, a, B, count, stream)
                    : launch_pipe_grouped<OP_MOD, false, false, EX>(dev, dtype, a, B, count, stream);
  });
}

}  // namespace dit
