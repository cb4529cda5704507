// policy_table.h -- all-reduce policy per group size, written by
// collective_datapath_gb300/tune.py from measurements; do not edit by hand.
// measured on NVIDIA GB300, warm (CUDA graph) us per op, sizes 8 KiB - 64 MiB per rank
// Entries: bytes per rank up to max_bytes use (encoding, algorithm, path).
#pragma once

#include <cstdint>

namespace coll {

struct PolicyEntry {
  uint64_t max_bytes;
  int enc, algo, path;
  int ctas;  // launch shape of the one-launch path (0 = one CTA per SM)
};

constexpr PolicyEntry kPolicy2[] = {
    {16384ull, 2, 1, 1, 64},  // SENT/oneshot/fused/narrow
    {32768ull, 0, 1, 1, 64},  // LL8/oneshot/fused/narrow
    {131072ull, 2, 1, 1, 64},  // SENT/oneshot/fused/narrow
    {344064ull, 2, 1, 1, 0},  // SENT/oneshot/fused
    {7421952ull, 2, 1, 1, 1024},  // SENT/oneshot/fused/wide
    {8421376ull, 2, 1, 2, 0},  // SENT/oneshot/streamed
    {UINT64_MAX, 1, 2, 3, 0},  // LL128/twoshot/composed
};
constexpr PolicyEntry kPolicy4[] = {
    {32768ull, 0, 1, 1, 64},  // LL8/oneshot/fused/narrow
    {65536ull, 2, 1, 1, 64},  // SENT/oneshot/fused/narrow
    {245760ull, 2, 1, 1, 0},  // SENT/oneshot/fused
    {524288ull, 2, 1, 1, 1024},  // SENT/oneshot/fused/wide
    {1982464ull, 1, 2, 3, 0},  // LL128/twoshot/composed
    {4456448ull, 2, 2, 1, 1024},  // SENT/twoshot/fused/wide
    {UINT64_MAX, 1, 2, 3, 0},  // LL128/twoshot/composed
};
constexpr PolicyEntry kPolicy8[] = {
    {16384ull, 0, 1, 1, 64},  // LL8/oneshot/fused/narrow
    {32768ull, 0, 1, 1, 0},  // LL8/oneshot/fused
    {65536ull, 2, 1, 1, 0},  // SENT/oneshot/fused
    {311296ull, 2, 1, 1, 1024},  // SENT/oneshot/fused/wide
    {1769472ull, 1, 2, 3, 0},  // LL128/twoshot/composed
    {2097152ull, 2, 2, 1, 1024},  // SENT/twoshot/fused/wide
    {UINT64_MAX, 1, 2, 3, 0},  // LL128/twoshot/composed
};

// group sizes with a table, in increasing order
constexpr int kPolicyGroups[] = {2, 4, 8};

inline const PolicyEntry* policy_table(int group, int* len) {
  switch (group) {
    case 2: *len = (int)(sizeof(kPolicy2) / sizeof(PolicyEntry)); return kPolicy2;
    case 4: *len = (int)(sizeof(kPolicy4) / sizeof(PolicyEntry)); return kPolicy4;
    case 8: *len = (int)(sizeof(kPolicy8) / sizeof(PolicyEntry)); return kPolicy8;
    default: *len = 0; return nullptr;
  }
}

}  // namespace coll
