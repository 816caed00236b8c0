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
DIT_WROW_SIG(OP_MOD, false, false, false, false);
#elif DIT_INSTANCE == 1
DIT_WROW_SIG(OP_MOD, false, true, false, false);
#elif DIT_INSTANCE == 2
DIT_WROW_SIG(OP_FUSED, false, false, false, false);
#elif DIT_INSTANCE == 3
DIT_WROW_SIG(OP_FUSED, false, true, false, false);
#elif DIT_INSTANCE == 4
DIT_WROW_SIG(OP_MOD, false, false, false, true);
#elif DIT_INSTANCE == 5
DIT_WROW_SIG(OP_MOD, false, true, false, true);
#elif DIT_INSTANCE == 6
DIT_WROW_SIG(OP_FUSED, false, false, false, true);
#elif DIT_INSTANCE == 7
DIT_WROW_SIG(OP_FUSED, false, true, false, true);
#elif DIT_INSTANCE == 8
DIT_PIPE_SIG(OP_MOD, false, false, false, false);
#elif DIT_INSTANCE == 9
DIT_PIPE_SIG(OP_MOD, false, true, false, false);
#elif DIT_INSTANCE == 10
DIT_PIPE_SIG(OP_MOD, false, false, true, false);
#elif DIT_INSTANCE == 11
DIT_PIPE_SIG(OP_MOD, false, true, true, false);
#elif DIT_INSTANCE == 12
DIT_PIPE_SIG(OP_FUSED, false, false, false, false);
#elif DIT_INSTANCE == 13
DIT_PIPE_SIG(OP_FUSED, false, true, false, false);
#elif DIT_INSTANCE == 14
DIT_PIPE_SIG(OP_FUSED, true, false, false, false);
#elif DIT_INSTANCE == 15
DIT_PIPE_SIG(OP_FUSED, true, true, false, false);
#elif DIT_INSTANCE == 16
DIT_PIPE_SIG(OP_FUSED, false, false, true, false);
#elif DIT_INSTANCE == 17
DIT_PIPE_SIG(OP_FUSED, false, true, true, false);
#elif DIT_INSTANCE == 18
DIT_PIPE_SIG(OP_FUSED, true, false, true, false);
#elif DIT_INSTANCE == 19
DIT_PIPE_SIG(OP_FUSED, true, true, true, false);
#elif DIT_INSTANCE == 20
DIT_PIPE_SIG(OP_MOD, false, false, false, true);
#elif DIT_INSTANCE == 21
DIT_PIPE_SIG(OP_MOD, false, true, false, true);
#elif DIT_INSTANCE == 22
DIT_PIPE_SIG(OP_MOD, false, false, true, true);
#elif DIT_INSTANCE == 23
DIT_PIPE_SIG(OP_MOD, false, true, true, true);
#elif DIT_INSTANCE == 24
DIT_PIPE_SIG(OP_FUSED, false, false, false, true);
#elif DIT_INSTANCE == 25
DIT_PIPE_SIG(OP_FUSED, false, true, false, true);
#elif DIT_INSTANCE == 26
DIT_PIPE_SIG(OP_FUSED, true, false, false, true);
#elif DIT_INSTANCE == 27
DIT_PIPE_SIG(OP_FUSED, true, true, false, true);
#elif DIT_INSTANCE == 28
DIT_PIPE_SIG(OP_FUSED, false, false, true, true);
#elif DIT_INSTANCE == 29
DIT_PIPE_SIG(OP_FUSED, false, true, true, true);
#elif DIT_INSTANCE == 30
DIT_PIPE_SIG(OP_FUSED, true, false, true, true);
#elif DIT_INSTANCE == 31
DIT_PIPE_SIG(OP_FUSED, true, true, true, true);
#elif DIT_INSTANCE == 32
DIT_GROUPED_SIG(OP_RGA, false, false, false);
DIT_GROUPED_SIG(OP_MOD, false, false, false);
DIT_GROUPED_SIG(OP_MOD, false, true, false);
#elif DIT_INSTANCE == 33
DIT_GROUPED_SIG(OP_MOD, false, false, true);
DIT_GROUPED_SIG(OP_MOD, false, true, true);
#elif DIT_INSTANCE == 34
DIT_GROUPED_SIG(OP_FUSED, false, false, false);
DIT_GROUPED_SIG(OP_FUSED, false, true, false);
#elif DIT_INSTANCE == 35
DIT_GROUPED_SIG(OP_FUSED, true, false, false);
DIT_GROUPED_SIG(OP_FUSED, true, true, false);
#elif DIT_INSTANCE == 36
DIT_GROUPED_SIG(OP_FUSED, false, false, true);
DIT_GROUPED_SIG(OP_FUSED, false, true, true);
#elif DIT_INSTANCE == 37
DIT_GROUPED_SIG(OP_FUSED, true, false, true);
DIT_GROUPED_SIG(OP_FUSED, true, true, true);
#elif DIT_INSTANCE == 38
DIT_WROW_SIG(OP_MOD, false, false, true, true);
#elif DIT_INSTANCE == 39
DIT_WROW_SIG(OP_MOD, false, true, true, true);
#elif DIT_INSTANCE == 40
DIT_WROW_SIG(OP_FUSED, false, false, true, true);
#elif DIT_INSTANCE == 41
DIT_WROW_SIG(OP_FUSED, false, true, true, true);
#else
#error "no such instance group"
#endif

}  // namespace dit
