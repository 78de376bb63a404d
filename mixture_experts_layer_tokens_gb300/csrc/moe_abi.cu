// moe_abi: host-side helpers shared by the entry points -- status strings,
// the device status word, SM counts.
#include "moe_common.cuh"

namespace moe {

int num_sms() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (dev >= 0 && dev < 64 && cached[dev]) return cached[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 1;
  if (dev >= 0 && dev < 64) cached[dev] = n;
  return n;
}

bool fits_int32(long long v) { return v >= 0 && v < 2147483647LL; }

}  // namespace moe

using namespace moe;

extern "C" moe_status_t moe_device_status(int clear) {
  if (cudaDeviceSynchronize() != cudaSuccess) return MOE_ERR_CUDA;
  const moe_status_t a = experts_status(clear);
  const moe_status_t b = align_status(clear);
  const moe_status_t c = prepare_status(clear);
  const moe_status_t d = finalize_status(clear);
  return a != MOE_OK ? a : (b != MOE_OK ? b : (c != MOE_OK ? c : d));
}

extern "C" const char* moe_status_string(moe_status_t status) {
  switch (status) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported configuration";
    case MOE_ERR_WORKSPACE: return "workspace missing or too small";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_TIMEOUT: return "device-side wait timed out";
  }
  return "unknown status";
}
