// Tensor-core (tcgen05) backward pass.
#include "fa_internal.h"

fa_status fa_launch_bwd_tc(const FaBwdProblem &p) {
    (void)p;
    return FA_ERR_UNSUPPORTED;
}
