// k_fused.cu -- residual gate and RMSNorm-modulation in one pass on GB300.
//
// residual_out = hidden + update * gate (sglang PR #29361, Motivation), then
// modulated_out = rms_norm(residual_out, eps) * (1 + scale) + shift (prhub
// summary of sglang PR #34172, "key source snippet"), the statistic taken
// over the residual as stored.  The rounded residual stays on chip between
// its store and the modulation -- written back over the row's shared-memory
// slot in the staged kernels, held in registers in the register kernel -- so
// the row is read from HBM once (hidden, update, gate) and written twice
// (residual, modulated output).
// Kernels (chosen in dit_rows.cuh): two warps per row on large tensors with
// a [B, 1, D] gate (dit_wrow.cuh), the staged CTA-per-row kernel otherwise
// (dit_pipe.cuh), the register and two-pass kernels for unaligned or long
// rows.
#include "dit_rows.cuh"

namespace dit {

cudaError_t launch_fused(const DeviceInfo& dev, int dtype, int vb, bool gate_full,
                         bool mod_full, const RowArgs& a, int64_t B, cudaStream_t stream) {
  if (gate_full)
    return mod_full ? launch_row_op<OP_FUSED, true, true>(dev, dtype, vb, a, B, stream)
                    : launch_row_op<OP_FUSED, true, false>(dev, dtype, vb, a, B, stream);
  return mod_full ? launch_row_op<OP_FUSED, false, true>(dev, dtype, vb, a, B, stream)
                  : launch_row_op<OP_FUSED, false, false>(dev, dtype, vb, a, B, stream);
}

cudaError_t launch_fused_fp8(const DeviceInfo& dev, int dtype, bool gate_full, bool mod_full,
                             const RowArgs& a, int64_t B, cudaStream_t stream) {
  return with_statistic<OP_FUSED>(a.exact, [&](auto ex) {
    constexpr bool EX = decltype(ex)::value;
    if (gate_full)
      return mod_full ? launch_pipe<OP_FUSED, true, true, true, EX>(dev, dtype, a, B, stream)
                      : launch_pipe<OP_FUSED, true, false, true, EX>(dev, dtype, a, B, stream);
    if constexpr (EX) {
      // the exact statistic on large tensors: two warps per row (the staged
      // kernel's exact instantiation for E4M3 spills)
      const cudaError_t w =
          mod_full ? launch_wrow<OP_FUSED, false, true, true, true>(dev, dtype, a, B, stream)
                   : launch_wrow<OP_FUSED, false, false, true, true>(dev, dtype, a, B, stream);
      if (w != cudaErrorNotSupported) return w;
    }
    return mod_full ? launch_pipe<OP_FUSED, false, true, true, EX>(dev, dtype, a, B, stream)
                    : launch_pipe<OP_FUSED, false, false, true, EX>(dev, dtype, a, B, stream);
  });
}

cudaError_t launch_fused_grouped(const DeviceInfo& dev, int dtype, bool gate_full,
                                 bool mod_full, const RowArgs* a, const int64_t* B, int count,
                                 cudaStream_t stream) {
  return with_statistic<OP_FUSED>(count > 0 && a[0].exact, [&](auto ex) {
    constexpr bool EX = decltype(ex)::value;
    if (gate_full)
      return mod_full
                 ? launch_pipe_grouped<OP_FUSED, true, true, EX>(dev, dtype, a, B, count, stream)
                 : launch_pipe_grouped<OP_FUSED, true, false, EX>(dev, dtype, a, B, count, stream);
    return mod_full
               ? launch_pipe_grouped<OP_FUSED, false, true, EX>(dev, dtype, a, B, count, stream)
               : launch_pipe_grouped<OP_FUSED, false, false, EX>(dev, dtype, a, B, count, stream);
  });
}

}  // namespace dit
