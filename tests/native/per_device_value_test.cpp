// Host test of tq::PerDeviceValue (kernel attributes, SM counts and occupancy
// answers cached per device): values are kept per device, make() runs once per
// device even when threads race, failures are not cached, out-of-range
// devices are refused.  Built and run by tests/test_abi_host.py with g++.
#include <atomic>
#include <cstdio>
#include <thread>
#include <vector>

#include "tq_once.h"

#define CHECK(c)                                                   \
  do {                                                             \
    if (!(c)) {                                                    \
      std::printf("FAIL line %d: %s\n", __LINE__, #c);             \
      return 1;                                                    \
    }                                                              \
  } while (0)

int main() {
  tq::PerDeviceValue v;
  int calls = 0;
  CHECK(v.get(0, [&] { ++calls; return 152; }) == 152);
  CHECK(v.get(0, [&] { ++calls; return 7; }) == 152);  // cached for device 0
  CHECK(calls == 1);
  CHECK(v.get(1, [&] { ++calls; return 148; }) == 148);  // device 1 has its own
  CHECK(calls == 2);
  CHECK(v.get(0, [&] { return 1; }) == 152 && v.get(1, [&] { return 1; }) == 148);
  // a failed make() is returned, not cached
  CHECK(v.get(2, [&] { ++calls; return -3; }) == -3);
  CHECK(v.get(2, [&] { ++calls; return 5; }) == 5);
  CHECK(calls == 4);
  // devices outside the table are refused without calling make()
  CHECK(v.get(-1, [&] { ++calls; return 1; }) == -1);
  CHECK(v.get(tq::kMaxDevices, [&] { ++calls; return 1; }) == -1);
  CHECK(calls == 4);
  // threads racing on one device: make() runs once, all see its value
  tq::PerDeviceValue w;
  std::atomic<int> made{0};
  std::vector<int> seen(16, 0);
  std::vector<std::thread> th;
  for (int i = 0; i < 16; ++i)
    th.emplace_back([&, i] {
      seen[i] = w.get(3, [&] {
        made.fetch_add(1);
        std::this_thread::sleep_for(std::chrono::milliseconds(20));
        return 42;
      });
    });
  for (auto& t : th) t.join();
  CHECK(made.load() == 1);
  for (int i = 0; i < 16; ++i) CHECK(seen[i] == 42);
  std::printf("ok\n");
  return 0;
}
