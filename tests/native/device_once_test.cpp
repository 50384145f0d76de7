// Host-only check of sv::device_once (the per-device launch set-up of the
// library): the set-up runs once per device ordinal, separately for each
// device, not at all for a bad ordinal, again after a failure, and once when
// several threads race on a device.  Prints "ok" and exits 0 on success.
#include <cstdio>
#include <thread>
#include <vector>

#include "sv_once.h"

static int fails = 0;
#define CHECK(c)                                                        \
    do {                                                                \
        if (!(c)) {                                                     \
            std::printf("FAIL line %d: %s\n", __LINE__, #c);            \
            ++fails;                                                    \
        }                                                               \
    } while (0)

int main()
{
    sv::DeviceOnce once;
    int calls[sv::SV_MAX_DEVICES] = {};
    auto setup = [&](int dev, int* v) {
        ++calls[dev];
        *v = 100 + dev;
        return 0;
    };
    int v = -1;
    CHECK(sv::device_once(once, 0, 0, -1, &v, setup) == 0 && v == 100);
    CHECK(sv::device_once(once, 0, 0, -1, &v, setup) == 0 && v == 100);
    CHECK(calls[0] == 1);
    // a second device runs its own set-up and keeps its own value
    CHECK(sv::device_once(once, 1, 0, -1, &v, setup) == 0 && v == 101);
    CHECK(calls[1] == 1);
    CHECK(sv::device_once(once, 0, 0, -1, &v, setup) == 0 && v == 100);
    // ordinals outside the table are refused without a set-up
    CHECK(sv::device_once(once, -1, 0, -1, &v, setup) == -1);
    CHECK(sv::device_once(once, sv::SV_MAX_DEVICES, 0, -1, &v, setup) == -1);
    // a failed set-up is not recorded: the next call tries again
    int tries = 0;
    auto flaky = [&](int, int* w) {
        *w = 7;
        return ++tries == 1 ? 5 : 0;
    };
    CHECK(sv::device_once(once, 3, 0, -1, &v, flaky) == 5);
    CHECK(sv::device_once(once, 3, 0, -1, &v, flaky) == 0 && v == 7);
    CHECK(tries == 2);
    // racing threads: one set-up, every thread sees its value
    sv::DeviceOnce race;
    int race_calls = 0;
    std::vector<std::thread> th;
    std::vector<int> seen(16, -1);
    for (int t = 0; t < 16; ++t)
        th.emplace_back([&, t] {
            sv::device_once(race, 2, 0, -1, &seen[t], [&](int, int* w) {
                ++race_calls;  // under the lock
                *w = 42;
                return 0;
            });
        });
    for (auto& x : th) x.join();
    CHECK(race_calls == 1);
    for (int t = 0; t < 16; ++t) CHECK(seen[t] == 42);
    if (fails == 0) std::printf("ok\n");
    return fails == 0 ? 0 : 1;
}
