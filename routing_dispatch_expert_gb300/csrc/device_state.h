// Per-device host state of the library (plain C++; no CUDA types, so it can be checked on a host
// without a GPU).
//
// Launch attributes (cudaFuncSetAttribute), occupancy results, SM counts, library-owned streams and
// the device address of a static __device__ array all belong to one device, and to one context on it:
// cudaDeviceReset ends the primary context, and another context made current is a different one.
// PerDevice<T> keeps one value per device ordinal, tagged with the context it was set up under; the
// set-up runs the first time a call finds no value for the current (device, context), under a mutex,
// so concurrent host threads set a device up once and never read a half-written value.
#pragma once

#include <mutex>

namespace moe {

constexpr int kMaxDevices = 64;

template <class T>
class PerDevice {
 public:
  // *out = the value of device `dev` under context `ctx`, running init(T&) first if there is none yet
  // (or if it was set up under another context). init returns 0 on success; a failed init stores
  // nothing, so the next call retries it. Returns init's status, or -1 for an ordinal outside
  // [0, kMaxDevices).
  template <class Init>
  int get(int dev, const void* ctx, Init&& init, T* out) {
    if (dev < 0 || dev >= kMaxDevices) return -1;
    std::lock_guard<std::mutex> lock(mu_);
    Slot& s = slots_[dev];
    if (!s.ready || s.ctx != ctx) {
      T v{};
      const int rc = init(v);
      if (rc != 0) return rc;
      s.value = v;
      s.ctx = ctx;
      s.ready = true;
    }
    *out = s.value;
    return 0;
  }

  // how many devices hold a value (for tests)
  int ready_count() {
    std::lock_guard<std::mutex> lock(mu_);
    int n = 0;
    for (const Slot& s : slots_) n += s.ready ? 1 : 0;
    return n;
  }

 private:
  struct Slot {
    const void* ctx = nullptr;
    bool ready = false;
    T value{};
  };
  std::mutex mu_;
  Slot slots_[kMaxDevices];
};

}  // namespace moe
