// Library-internal host helpers of the attention calls (not part of the C ABI).
#pragma once
#include <stddef.h>

namespace pkv {

// Parts of the default partition for the current device: every SM holding as
// many CTAs of the variant for (D, dtype, flags, G = Hq / Hkv) as fit at once.
int default_parts(int D, int dtype, int flags, int G, int *parts);

// Leading bytes of an attention workspace that hold the fused merge's
// counters (the only bytes a call expects to find zero).
size_t workspace_counter_bytes(int B, int Hq, int Hkv, int D, int C);

}  // namespace pkv
