// Device-side status word shared by every kernel of the library.
//
// Kernels never trap. A wait that runs out of time, or a launch that finds an
// inconsistent configuration, ORs a bit into the status word whose address
// the host passes as a kernel argument; bea_get_device_status() reads and
// clears it.
#pragma once

#include <cstdint>

namespace bea {

enum : uint32_t {
  BEA_STATUS_TIMEOUT = 1u,  // an mbarrier wait ran past its limit
  BEA_STATUS_CONFIG = 2u,   // a kernel was launched with a configuration it cannot run
};

__device__ __forceinline__ void report_status(uint32_t* status, uint32_t code) {
  if (status != nullptr) atomicOr(status, code);
}

}  // namespace bea
