// vla_internal.h -- entry points shared by the library's translation units;
// not part of the C ABI (include/vla.h).
#pragma once

#include <stddef.h>

#include "vla.h"

namespace vla_impl {

// vla_forward_ex() with the rows of head h of o starting o_head_stride
// elements after those of head h - 1 (0 = T * d, the [B, H, T, d] layout of
// vla_forward). A larger stride lets a launch over tokens [t0, t0 + T) of a
// longer sequence write straight into that sequence's output array.
vla_status forward(const void* q, const void* k, const void* v, const void* u, vla_dtype dtype, int B, int H, int T,
                   int d, float lambda0, float eps, const float* S0, const float* A0, const float* zk0, float* o,
                   float* S_out, float* A_out, float* zk_out, void* workspace, size_t workspace_bytes, void* stream,
                   const vla_options* opts, size_t o_head_stride);

// Bytes of workspace every kernel choice needs at any valid shape (the status
// record): with only this much, VLA_ALGO_AUTO never takes the segmented path.
size_t status_bytes();

}  // namespace vla_impl
