// Host-only check of moe::PerDevice (the per-device launch state of the library): values are kept per
// device ordinal and per context, set up once per (device, context) even under concurrent threads,
// and a failed set-up is retried. Built and run by tests/test_device_state.py with g++ (no GPU).
#include <atomic>
#include <cstdio>
#include <thread>
#include <vector>

#include "device_state.h"

#define CHECK(c)                                              \
  do {                                                        \
    if (!(c)) {                                               \
      std::printf("FAILED line %d: %s\n", __LINE__, #c);      \
      return 1;                                               \
    }                                                         \
  } while (0)

int main() {
  moe::PerDevice<int> table;
  std::atomic<int> inits[moe::kMaxDevices];
  for (auto& a : inits) a = 0;
  int ctx_a = 0, ctx_b = 0;  // two distinct context handles

  // 8 threads x 4 devices, each thread asking every device many times: one set-up per device
  std::vector<std::thread> threads;
  std::atomic<int> bad{0};
  for (int t = 0; t < 8; ++t)
    threads.emplace_back([&] {
      for (int rep = 0; rep < 200; ++rep)
        for (int dev = 0; dev < 4; ++dev) {
          int v = -1;
          const int rc = table.get(dev, &ctx_a, [&](int& out) { inits[dev]++; out = 100 + dev; return 0; }, &v);
          if (rc != 0 || v != 100 + dev) bad++;
        }
    });
  for (auto& th : threads) th.join();
  CHECK(bad == 0);
  for (int dev = 0; dev < 4; ++dev) CHECK(inits[dev] == 1);
  CHECK(table.ready_count() == 4);

  // the value of one device does not leak into another
  int v = -1;
  CHECK(table.get(5, &ctx_a, [](int& out) { out = 7; return 0; }, &v) == 0 && v == 7);
  CHECK(table.get(2, &ctx_a, [](int& out) { out = -99; return 0; }, &v) == 0 && v == 102);

  // a new context on the same device sets the device up again
  CHECK(table.get(2, &ctx_b, [&](int& out) { inits[2]++; out = 202; return 0; }, &v) == 0 && v == 202);
  CHECK(inits[2] == 2);
  CHECK(table.get(2, &ctx_b, [&](int& out) { inits[2]++; out = -1; return 0; }, &v) == 0 && v == 202);
  CHECK(inits[2] == 2);

  // a failed set-up stores nothing and is retried by the next call
  CHECK(table.get(9, &ctx_a, [](int& out) { out = 1; return 17; }, &v) == 17);
  CHECK(table.get(9, &ctx_a, [](int& out) { out = 9; return 0; }, &v) == 0 && v == 9);

  // ordinals outside the table are rejected without running the set-up
  bool ran = false;
  CHECK(table.get(-1, &ctx_a, [&](int& out) { ran = true; out = 0; return 0; }, &v) == -1);
  CHECK(table.get(moe::kMaxDevices, &ctx_a, [&](int& out) { ran = true; out = 0; return 0; }, &v) == -1);
  CHECK(!ran);
  std::printf("ok\n");
  return 0;
}
