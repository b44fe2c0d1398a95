// Per-device one-time set-up (plain C++, no CUDA types).
//
// Kernel attributes such as the dynamic shared-memory limit, device symbol
// addresses and SM counts belong to one device.  A process-wide "once" would set
// them on the first device only and leave a second device of the same process at
// its defaults, so every such step runs once per device instead: the first call
// for a device runs the set-up (with that device current) and keeps its result,
// and later calls for that device return the kept result.
#pragma once

#include <mutex>
#include <vector>

namespace qcf {

template <typename Result>
class PerDevice {
 public:
  // Result of set_up() for device `dev`; set_up runs at most once per device.
  // A negative `dev` (the current device could not be read) is not cached.
  template <typename F>
  Result get(int dev, F&& set_up) {
    if (dev < 0) return set_up();
    std::lock_guard<std::mutex> lk(mu_);
    if (static_cast<size_t>(dev) >= done_.size()) {
      done_.resize(dev + 1, 0);
      value_.resize(dev + 1);
    }
    if (!done_[dev]) {
      value_[dev] = set_up();
      done_[dev] = 1;
    }
    return value_[dev];
  }

 private:
  std::mutex mu_;
  std::vector<char> done_;
  std::vector<Result> value_;
};

}  // namespace qcf
