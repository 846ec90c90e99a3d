// Per-device queries shared by the libttc translation units.
#include "ttc_internal.h"

namespace ttc {

int device_sms() {
  static std::mutex mu;
  static int sms[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 1;
  std::lock_guard<std::mutex> lock(mu);
  if (!sms[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 1;
    sms[dev] = n;
  }
  return sms[dev];
}

}  // namespace ttc
