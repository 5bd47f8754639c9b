// lr_sel_bf16_z_sp.cu -- one compiled variant of the selective scan kernel:
// bf16 I/O, with the silu(z) gate, softplus applied to dt (see lr_selective.cuh).
#include "lr_selective.cuh"

namespace lr {
namespace sel {
LR_SEL_DEFINE(bf16_z_sp, __nv_bfloat16, false, true, true)
}  // namespace sel
}  // namespace lr
