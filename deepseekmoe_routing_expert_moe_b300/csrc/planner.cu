// Redundant-expert placement from the load histogram ("02 · DeepSeek-V3"
// §5.1: high-load experts are replicated from online load statistics -- 32
// redundant experts, one extra expert per GPU for prefill -- and the set is
// revised periodically).  Host code: it runs between steps on a count
// vector the caller has read back (moe_forward's counts_out, summed over
// the statistics window), not on the layer's device path.
//
// Base placement: device d hosts experts [d*E/D, (d+1)*E/D).  An expert
// with a copy serves its c tokens round-robin, the original keeping
// ceil(c/2) and the copy floor(c/2).  Walking the experts heaviest first
// (load desc, index asc) while slots are free and loads positive, each gets
// a copy on the least-loaded device (ties: lower index) that has a free
// slot and is not its own; an expert whose only free slots are on its own
// device is passed over.
#include <algorithm>
#include <cstdint>
#include <numeric>
#include <vector>

#include "../../include/moe.h"

extern "C" moe_status_t moe_plan_redundant_experts(
    const int64_t* load, int32_t E, int32_t n_devices,
    int32_t slots_per_device, int32_t* slot_expert, int64_t* device_load) {
  if (load == nullptr || device_load == nullptr || E <= 0 ||
      n_devices <= 0 || slots_per_device < 0 || E % n_devices != 0)
    return MOE_ERR_INVALID_ARG;
  const long long R = (long long)n_devices * slots_per_device;
  if (R > 0 && slot_expert == nullptr) return MOE_ERR_INVALID_ARG;
  for (int32_t e = 0; e < E; ++e)
    if (load[e] < 0) return MOE_ERR_INVALID_ARG;
  const int32_t per = E / n_devices;
  std::vector<int64_t> dev(n_devices, 0);
  for (int32_t e = 0; e < E; ++e) dev[e / per] += load[e];
  std::vector<int32_t> used(n_devices, 0);
  for (long long i = 0; i < R; ++i) slot_expert[i] = -1;

  std::vector<int32_t> order(E);
  std::iota(order.begin(), order.end(), 0);
  std::stable_sort(order.begin(), order.end(), [&](int32_t a, int32_t b) {
    return load[a] > load[b];  // stable: equal loads keep index order
  });
  long long free_slots = R;
  for (int32_t e : order) {
    if (free_slots == 0 || load[e] <= 0) break;
    const int32_t home = e / per;
    int32_t best = -1;
    for (int32_t d = 0; d < n_devices; ++d) {
      if (d == home || used[d] >= slots_per_device) continue;
      if (best < 0 || dev[d] < dev[best]) best = d;
    }
    if (best < 0) continue;  // only its own device has a free slot
    const int64_t share = load[e] / 2;
    dev[home] -= share;
    dev[best] += share;
    slot_expert[(long long)best * slots_per_device + used[best]] = e;
    ++used[best];
    --free_slots;
  }
  std::copy(dev.begin(), dev.end(), device_load);
  return MOE_OK;
}
