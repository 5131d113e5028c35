// Values that the library sets up once per CUDA device: a kernel's opt-in to
// more than 48 KB of dynamic shared memory, a device's SM count, how many SM
// pairs a clustered kernel can keep resident.  CUDA keeps function attributes
// and device properties per device, so a process that drives several GPUs
// needs each of them once for every device it launches on; a single
// process-wide flag would leave the second GPU's launches without the
// opt-in.  Host code only (no CUDA types), so the keying can be tested on a
// machine without a GPU.
#pragma once

#include <mutex>

namespace fp8q {

constexpr int kMaxDevices = 64;

// One value of type T per device ordinal, filled on first use by `fill`
// (which returns false on failure, leaving the slot empty so that a later
// call retries).  Safe to call from several host threads.
template <typename T>
class PerDevice {
   public:
    template <typename F>
    bool get(int dev, T& out, F&& fill) {
        if (dev < 0 || dev >= kMaxDevices) return false;
        std::lock_guard<std::mutex> lock(mu_);
        if (!set_[dev]) {
            T v{};
            if (!fill(v)) return false;
            val_[dev] = v;
            set_[dev] = true;
        }
        out = val_[dev];
        return true;
    }

   private:
    std::mutex mu_;
    bool set_[kMaxDevices] = {};
    T val_[kMaxDevices] = {};
};

}  // namespace fp8q
