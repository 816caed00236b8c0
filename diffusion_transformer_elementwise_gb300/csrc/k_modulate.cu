// k_modulate.cu -- out = rms_norm(x, eps) * (1 + scale) + shift on GB300.
//
// Operation: prhub summary of sglang PR #34172 (LTX-2 quality=high fused
// RMSNorm+modulate), section "key source snippet" (the expression of
// _ltx2_rms_norm_modulate) and section "implementation breakdown", item 2
// (weightless RMSNormNoWeight, the whole expression in one launch).
//
// [B, 1, D] scale/shift on 16-byte aligned rows: one warp per row
// (dit_warprow.cuh), no CTA barrier per row.  [B, L, D] scale/shift, or rows
// too long for that kernel's shared memory: the CTA-per-row staged kernel
// (dit_pipe.cuh).  Unaligned rows: the register kernel (dit_rows.cuh).
#include "dit_rows.cuh"
#include "dit_warprow.cuh"

namespace dit {

cudaError_t launch_modulate(const DeviceInfo& dev, int dtype, int vb, bool mod_full,
                            const RowArgs& a, int64_t B, cudaStream_t stream) {
#ifndef DIT_NO_WARP_ROWS  // tuning builds: the CTA-per-row kernel only
  if (!mod_full && vb >= 16) {
    const cudaError_t e = dispatch_dtype_width(dtype, 16, [&](auto tt, auto) -> cudaError_t {
      using T = typename decltype(tt)::type;
      return launch_warp_mod<T>(dev, a, B, stream);
    });
    if (e != cudaErrorNotSupported) return e;
  }
#endif
  return mod_full ? launch_row_op<OP_MOD, false, true>(dev, dtype, vb, a, B, stream)
                  : launch_row_op<OP_MOD, false, false>(dev, dtype, vb, a, B, stream);
}

}  // namespace dit
