// draft_tc.cu -- tensor-core Markov draft (not yet enabled).
#include "draft_tc.cuh"

namespace dspark {

bool draft_tc_supported(int, int, int, int, int) { return false; }
size_t draft_tc_workspace(int, int, int) { return 0; }
int launch_draft_tc(const DraftTcArgs&, cudaStream_t) { return DSPARK_ERR_UNSUPPORTED; }

}  // namespace dspark
