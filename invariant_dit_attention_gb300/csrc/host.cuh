// host.cuh -- host-side state shared by every launcher of libh3attn: the
// driver's tensor-map encoder, per-device preparation (kernel attributes, SM
// count) and the rotary table built from a configuration.
#pragma once

#include <cudaTypedefs.h>

#include "common.cuh"

namespace h3 {

// The driver's cuTensorMapEncodeTiled, resolved once per process (thread-safe);
// null if the driver does not provide it.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();

// Prepares the current device once (thread-safe): checks that it is an sm_103
// GPU, sets the dynamic shared-memory limits of the tensor-core kernels and
// records its SM count.  cudaErrorNotSupported for another device or without
// the tensor-map encoder.
cudaError_t prepare_device();

// SM count of the current device, recorded by prepare_device() (0 if the
// device was not prepared).
int device_sms();

// Rotary layout of a configuration: sections of the t, h, w axes (each a
// multiple of 8, sum <= 128), base theta; rotate-half pairs inside a section,
// pair j of an n-channel axis turning at theta^(-2j/n).  False if the sections
// are not supported.
bool build_rope_table(const int sections[3], float theta, RopeTable& rt);

// Per-file parts of prepare_device (dynamic shared-memory limits).
cudaError_t set_fwd_attributes();
cudaError_t set_bwd_attributes();
cudaError_t set_linear_attributes();

}  // namespace h3
