// CUDA-core variants of the split-KV paged decode attention kernel, bf16 cache.
#include "attention_kernel.cuh"

namespace pkv {

bool attn_variant_simt_bf16(int D, int G, AttnVariant *v) {
  using T = __nv_bfloat16;
  if (G <= 2) G = 2;
  if (D == 64) {
    if (G == 2) { *v = AttnLauncher<T, 64, 4, 16, 1, 2>::variant(); return true; }
    if (G == 4) { *v = AttnLauncher<T, 64, 4, 16, 1, 4>::variant(); return true; }
    if (G == 8) { *v = AttnLauncher<T, 64, 4, 16, 1, 8>::variant(); return true; }
  } else if (D == 128) {
    if (G == 2) { *v = AttnLauncher<T, 128, 4, 8, 1, 2>::variant(); return true; }
    if (G == 4) { *v = AttnLauncher<T, 128, 4, 8, 1, 4>::variant(); return true; }
    if (G == 8) { *v = AttnLauncher<T, 128, 4, 8, 1, 8>::variant(); return true; }
  }
  return false;
}

}  // namespace pkv
