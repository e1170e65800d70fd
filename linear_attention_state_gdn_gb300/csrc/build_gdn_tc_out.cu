// build_gdn_tc_out.cu -- the outputs instance of the DeltaNet / GDN chain kernel (see the
// header of build_gdn_tc.cu), compiled in a translation unit of its own so that the plain
// chain's code is the same as without it.
#define HYPIC_GDN_TC_OUTPUTS 1
#include "build_gdn_tc.cu"
