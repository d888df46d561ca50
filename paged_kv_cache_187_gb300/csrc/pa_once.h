// pa_once.h -- once-per-device set-up bookkeeping for the kernel launchers (plain C++,
// no CUDA, so that it also compiles into a host-only test).
#pragma once

#include <bitset>
#include <mutex>

namespace pa {

// Remembers, per device ordinal, whether a set-up step (a kernel attribute, which the
// CUDA runtime keeps per device) has succeeded there.  run(dev, f) calls f() on the first
// call for `dev` and on every later call until f() returns 0 (success); after that it
// returns 0 without calling f.  Ordinals beyond kMaxDevices call f() every time.  Safe to
// call from several threads: f runs under the object's lock.
class PerDeviceOnce {
public:
    static constexpr int kMaxDevices = 256;

    template <class F>
    int run(int dev, F&& f) {
        if (dev < 0 || dev >= kMaxDevices) return static_cast<int>(f());
        std::lock_guard<std::mutex> lk(mu_);
        if (done_[dev]) return 0;
        const int e = static_cast<int>(f());
        if (e == 0) done_[dev] = true;
        return e;
    }

    bool done(int dev) {
        if (dev < 0 || dev >= kMaxDevices) return false;
        std::lock_guard<std::mutex> lk(mu_);
        return done_[dev];
    }

private:
    std::mutex mu_;
    std::bitset<kMaxDevices> done_;
};

}  // namespace pa
