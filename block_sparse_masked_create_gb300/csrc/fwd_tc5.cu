// placeholder: replaced by the tcgen05 forward kernel
#include "fa_launch.h"
namespace fa {
int launch_fwd_tc5(const FwdArgs&, cudaStream_t) { return FA_ERR_UNSUPPORTED; }
}
