// Library-internal host helpers of the attention calls (not part of the C ABI).
#pragma once
#include <stddef.h>

namespace pkv {

// Pages of streaming a unit boundary costs a CTA (segment combine, pipeline
// drain), which the page-balanced partition charges per unit: measured on
// GB300 at ~0.7 us against ~0.17 us per page at d = 64 and ~0.33 us at d = 128.
inline int seg_cost(int D) { return D <= 64 ? 4 : 2; }

// Parts of the default partition for the current device: every SM holding as
// many CTAs of the variant for (D, dtype, flags, G = Hq / Hkv) as fit at once.
int default_parts(int D, int dtype, int flags, int G, int *parts);

// Leading bytes of an attention workspace that hold the fused merge's
// counters (the only bytes a call expects to find zero).
size_t workspace_counter_bytes(int B, int Hq, int Hkv, int D, int C);

// Shape rules every attention call checks (dtype, head size, B, the group
// size Hq / Hkv); PKV_OK or the error, with the message set.
int check_shapes(int B, int Hq, int Hkv, int D, int dtype);

}  // namespace pkv
