// sv_once.h -- one-time launch set-up kept per device (plain C++, no CUDA).
//
// A kernel attribute (the dynamic shared-memory opt-in) and an occupancy
// query belong to one device: a process that runs the library on device 0
// and then on device 1 must repeat them there.  DeviceOnce records, per
// device ordinal, whether the set-up ran and the value it produced.  The
// first call for a device runs the set-up under a lock; every later call
// for that device reads the recorded value without locking.  A set-up that
// fails is not recorded, so the next call tries again.
#pragma once

#include <atomic>
#include <mutex>

namespace sv {

constexpr int SV_MAX_DEVICES = 64;

struct DeviceOnce {
    std::mutex mu;
    std::atomic<int> done[SV_MAX_DEVICES] = {};
    int value[SV_MAX_DEVICES] = {};
};

// Runs setup(dev, &value) once for device `dev`; returns its status
// (ok_status when it ran before) and stores the recorded value in *value.
// Status is any type whose ok_status compares equal on success.
template <typename Status, typename F>
Status device_once(DeviceOnce& o, int dev, Status ok_status, Status bad_device, int* value, F setup)
{
    if (dev < 0 || dev >= SV_MAX_DEVICES) return bad_device;
    if (o.done[dev].load(std::memory_order_acquire)) {
        if (value) *value = o.value[dev];
        return ok_status;
    }
    std::lock_guard<std::mutex> lock(o.mu);
    if (!o.done[dev].load(std::memory_order_relaxed)) {
        int v = 0;
        const Status st = setup(dev, &v);
        if (!(st == ok_status)) return st;
        o.value[dev] = v;
        o.done[dev].store(1, std::memory_order_release);
    }
    if (value) *value = o.value[dev];
    return ok_status;
}

}  // namespace sv
