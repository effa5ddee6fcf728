// Tensor-core (mma.sync, bf16 in / f32 accumulate) variants of the split-KV
// paged decode attention kernel.
#include "attention_kernel.cuh"

namespace pkv {

bool attn_variant_mma(int D, AttnVariant *v) {
  switch (D) {
    case 64: *v = AttnLauncher<__nv_bfloat16, 64, 4, 16, 0, 8>::variant(); return true;
    case 128: *v = AttnLauncher<__nv_bfloat16, 128, 4, 8, 0, 8>::variant(); return true;
    default: return false;
  }
}

}  // namespace pkv
