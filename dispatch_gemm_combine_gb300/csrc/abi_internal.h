// Helpers that more than one translation unit of the C ABI shares: the
// shape check, the per-device capability cache and launch accounting
// (the launch counter and the optional event timer of moe.h).  Not part of
// the C ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "moe.h"

namespace moe {

// moe_shape validity, as every entry point checks it.
bool abi_shape_ok(const moe_shape* s);

// SM count of the current device, or MOE_ERR_UNSUPPORTED if it is not an
// sm_103 part (cached per device).
moe_status abi_device_sms(int* sms);

// The plan kernels (launch_plan) and a memset, counted by
// moe_kernel_launch_count() and bracketed by the event timer when it is on.
cudaError_t abi_tracked_plan(const int* idx, int64_t Tk, int E, int* counts, int* offsets,
                             int* perm, int* inv, int* poff, int* blkhist, int* err,
                             cudaStream_t st);
cudaError_t abi_tracked_memset(void* p, int value, size_t bytes, cudaStream_t st);

}  // namespace moe
