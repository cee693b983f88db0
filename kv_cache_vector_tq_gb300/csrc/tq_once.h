// Values that belong to one device (its SM count, whether a kernel attribute
// has been set on it, how many CTAs of a kernel it holds per SM), made once per
// device and usable from several host threads.  Plain C++ (no CUDA types), so
// that the host tests can compile it alone.
#pragma once

#include <atomic>
#include <mutex>

namespace tq {

constexpr int kMaxDevices = 64;

// get(dev, make) returns the value cached for device `dev`, or calls make()
// (under a lock, so only once even when threads race) the first time.  A value
// <= 0 means make() failed: it is returned but not cached, so the next call
// tries again.  Devices outside [0, kMaxDevices) get -1 without calling make().
class PerDeviceValue {
 public:
  template <class Make>
  int get(int dev, Make&& make) {
    if (dev < 0 || dev >= kMaxDevices) return -1;
    int v = val_[dev].load(std::memory_order_acquire);
    if (v > 0) return v;
    std::lock_guard<std::mutex> lock(mu_);
    v = val_[dev].load(std::memory_order_relaxed);
    if (v > 0) return v;
    v = make();
    if (v > 0) val_[dev].store(v, std::memory_order_release);
    return v;
  }

 private:
  std::atomic<int> val_[kMaxDevices] = {};
  std::mutex mu_;
};

}  // namespace tq
