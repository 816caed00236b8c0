// k_instances.cu -- the row launchers' explicit instantiations.
//
// Each launcher instantiates a kernel per dtype and shape variant; together
// they are most of the library's compile time.  This file is compiled once
// for each value of DIT_INSTANCE (the build passes -DDIT_INSTANCE=k for every
// k below), one launcher -- or a few small ones -- per compilation, so they
// build in parallel.  dit_wrow.cuh and dit_pipe.cuh declare them extern for
// every other translation unit.
#include "dit_rows.cuh"

#ifndef DIT_INSTANCE
#error "k_instances.cu is compiled with -DDIT_INSTANCE=<k>"
#endif

namespace dit {

#if DIT_INSTANCE == 0
DIT_WROW_SIG(OP_MOD, false, false, false);
#elif DIT_INSTANCE == 1
DIT_WROW_SIG(OP_MOD, false, true, false);
#elif DIT_INSTANCE == 2
DIT_WROW_SIG(OP_FUSED, false, false, false);
#elif DIT_INSTANCE == 3
DIT_WROW_SIG(OP_FUSED, false, true, false);
#elif DIT_INSTANCE == 4
DIT_WROW_SIG(OP_FUSED, true, false, false);
#elif DIT_INSTANCE == 5
DIT_WROW_SIG(OP_FUSED, true, true, false);
#elif DIT_INSTANCE == 6
DIT_PIPE_SIG(OP_MOD, false, false, false);
#elif DIT_INSTANCE == 7
DIT_PIPE_SIG(OP_MOD, false, true, false);
#elif DIT_INSTANCE == 8
DIT_PIPE_SIG(OP_MOD, false, false, true);
#elif DIT_INSTANCE == 9
DIT_PIPE_SIG(OP_MOD, false, true, true);
#elif DIT_INSTANCE == 10
DIT_PIPE_SIG(OP_FUSED, false, false, false);
#elif DIT_INSTANCE == 11
DIT_PIPE_SIG(OP_FUSED, false, true, false);
#elif DIT_INSTANCE == 12
DIT_PIPE_SIG(OP_FUSED, true, false, false);
#elif DIT_INSTANCE == 13
DIT_PIPE_SIG(OP_FUSED, true, true, false);
#elif DIT_INSTANCE == 14
DIT_PIPE_SIG(OP_FUSED, false, false, true);
#elif DIT_INSTANCE == 15
DIT_PIPE_SIG(OP_FUSED, false, true, true);
#elif DIT_INSTANCE == 16
DIT_PIPE_SIG(OP_FUSED, true, false, true);
#elif DIT_INSTANCE == 17
DIT_PIPE_SIG(OP_FUSED, true, true, true);
#elif DIT_INSTANCE == 18
DIT_GROUPED_SIG(OP_RGA, false, false);
DIT_GROUPED_SIG(OP_MOD, false, false);
DIT_GROUPED_SIG(OP_MOD, false, true);
#elif DIT_INSTANCE == 19
DIT_GROUPED_SIG(OP_FUSED, false, false);
DIT_GROUPED_SIG(OP_FUSED, false, true);
#elif DIT_INSTANCE == 20
DIT_GROUPED_SIG(OP_FUSED, true, false);
DIT_GROUPED_SIG(OP_FUSED, true, true);
#else
#error "no such instance group"
#endif

}  // namespace dit
