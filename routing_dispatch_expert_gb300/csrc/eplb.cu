// Expert placement with redundant replicas (host side).
//
// Inference guide 6.4 "Data parallelism and expert parallelism", section 5.2 (the load simulation and
// its placement) and 5.3 (EPLB: redundant experts plus periodic rebalancing): the layer is as slow as
// its busiest card, so the hottest experts get extra replicas -- each extra replica goes to the expert
// with the highest load per replica -- and the replicas are then placed heaviest first, each onto the
// currently lightest card that still has a free slot. The plan is a table of physical slots (card-major,
// (E + R) / n_cards slots per card), each naming the logical expert whose weights it serves; dispatch
// spreads an expert's tokens round-robin over its replicas.
#include <stdint.h>

#include <algorithm>
#include <string>
#include <vector>

#include "../../include/moe.h"
#include "kernels.h"

namespace moe {

int eplb_plan(const int64_t* load, int E, int n_cards, int n_redundant, int32_t* replicas, int32_t* slot_expert,
              int32_t* slot_replica, int32_t* replica_slot, double* card_load, std::string* err) {
  if (!load || !replicas || !slot_expert || !slot_replica || !replica_slot || !card_load) {
    *err = "moe_eplb_plan: NULL argument";
    return MOE_ERR_INVALID;
  }
  if (E <= 0 || n_cards <= 0 || n_redundant < 0 || (E + n_redundant) % n_cards != 0) {
    *err = "moe_eplb_plan: need E > 0, n_cards > 0, n_redundant >= 0 and (E + n_redundant) % n_cards == 0";
    return MOE_ERR_INVALID;
  }
  // 1. redundant replicas: each goes to the expert with the largest load per replica (first on ties)
  for (int e = 0; e < E; ++e) replicas[e] = 1;
  for (int r = 0; r < n_redundant; ++r) {
    int best = 0;
    for (int e = 1; e < E; ++e)
      if ((double)load[e] / replicas[e] > (double)load[best] / replicas[best]) best = e;
    replicas[best] += 1;
  }
  // 2. every replica carries load / replicas; heaviest first, equal loads in expert order
  struct Copy {
    double w;
    int e;
  };
  std::vector<Copy> copies;
  copies.reserve(E + n_redundant);
  for (int e = 0; e < E; ++e)
    for (int i = 0; i < replicas[e]; ++i) copies.push_back({(double)load[e] / replicas[e], e});
  std::stable_sort(copies.begin(), copies.end(), [](const Copy& a, const Copy& b) { return a.w > b.w; });
  // 3. each onto the lightest card with a free slot (lowest card index on ties)
  const int per_card = (E + n_redundant) / n_cards;
  const int max_rep = n_redundant + 1;
  std::vector<int> used(n_cards, 0), placed(E, 0);
  for (int c = 0; c < n_cards; ++c) card_load[c] = 0.0;
  for (int i = 0; i < E * max_rep; ++i) replica_slot[i] = -1;
  for (const Copy& cp : copies) {
    int g = -1;
    for (int c = 0; c < n_cards; ++c)
      if (used[c] < per_card && (g < 0 || card_load[c] < card_load[g])) g = c;
    const int slot = g * per_card + used[g];
    slot_expert[slot] = cp.e;
    slot_replica[slot] = placed[cp.e];
    replica_slot[cp.e * max_rep + placed[cp.e]] = slot;
    placed[cp.e] += 1;
    used[g] += 1;
    card_load[g] += cp.w;
  }
  return MOE_OK;
}

}  // namespace moe
