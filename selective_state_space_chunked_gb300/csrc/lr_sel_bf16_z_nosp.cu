// lr_sel_bf16_z_nosp.cu -- one compiled variant of the selective scan kernel:
// bf16 I/O, with the silu(z) gate, dt taken as delta (see lr_selective.cuh).
#include "lr_selective.cuh"

namespace lr {
namespace sel {
LR_SEL_DEFINE(bf16_z_nosp, __nv_bfloat16, false, true, false)
}  // namespace sel
}  // namespace lr
