// build_gdn_tc_kda.cu -- the channel-gated (KDA) instance of the delta-rule chain kernel (see the
// header of build_gdn_tc.cu), compiled in a translation unit of its own so that the plain
// chain's code is the same as without it.
#define HYPIC_GDN_TC_KDA 1
#include "build_gdn_tc.cu"
