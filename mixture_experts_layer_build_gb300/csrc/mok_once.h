// mok_once.h -- one-time set-up per device (plain C++, no CUDA types, so host tests can drive it).
//
// A kernel attribute such as the dynamic shared-memory limit belongs to the device that is current
// when it is set: a process that drives several GPUs must set it once on each.  DeviceOnce runs a
// set-up step once per device id, under a lock, and remembers success only: a failed step is
// retried by the next call.  After the first success on a device the check is one atomic load.
#pragma once
#include <atomic>
#include <cstdint>
#include <mutex>

namespace mok {

class DeviceOnce {
 public:
  static constexpr int kMaxDevices = 64;

  // get_device(int*) -> 0 on success; setup() -> 0 on success.  Returns the first non-zero code
  // of either (a device id outside [0, 64) gives `bad_device`), else 0.
  template <class GetDevice, class Setup>
  int run(GetDevice&& get_device, Setup&& setup, int bad_device) {
    int dev = -1;
    const int rc = get_device(&dev);
    if (rc != 0) return rc;
    if (dev < 0 || dev >= kMaxDevices) return bad_device;
    const uint64_t bit = uint64_t(1) << dev;
    if (done_.load(std::memory_order_acquire) & bit) return 0;
    std::lock_guard<std::mutex> lk(mu_);
    if (done_.load(std::memory_order_relaxed) & bit) return 0;
    const int s = setup();
    if (s == 0) done_.fetch_or(bit, std::memory_order_release);
    return s;
  }

 private:
  std::mutex mu_;
  std::atomic<uint64_t> done_{0};
};

}  // namespace mok
