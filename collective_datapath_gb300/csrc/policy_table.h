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
    {65536ull, 0, 1, 1, 64},  // LL8/oneshot/fused/narrow
    {131072ull, 2, 1, 1, 64},  // SENT/oneshot/fused/narrow
    {770048ull, 2, 1, 1, 0},  // SENT/oneshot/fused
    {2998272ull, 2, 1, 1, 1024},  // SENT/oneshot/fused/wide
    {7421952ull, 2, 2, 1, 1024},  // SENT/twoshot/fused/wide
    {17432576ull, 1, 1, 2, 0},  // LL128/oneshot/streamed
    {UINT64_MAX, 1, 2, 2, 0},  // LL128/twoshot/streamed
};
constexpr PolicyEntry kPolicy4[] = {
    {32768ull, 0, 1, 1, 64},  // LL8/oneshot/fused/narrow
    {311296ull, 2, 1, 1, 0},  // SENT/oneshot/fused
    {983040ull, 2, 1, 1, 1024},  // SENT/oneshot/fused/wide
    {1900544ull, 2, 2, 1, 0},  // SENT/twoshot/fused
    {7421952ull, 2, 2, 1, 1024},  // SENT/twoshot/fused/wide
    {9109504ull, 1, 1, 2, 0},  // LL128/oneshot/streamed
    {UINT64_MAX, 1, 2, 2, 0},  // LL128/twoshot/streamed
};
constexpr PolicyEntry kPolicy8[] = {
    {8192ull, 0, 1, 1, 64},  // LL8/oneshot/fused/narrow
    {32768ull, 2, 1, 1, 64},  // SENT/oneshot/fused/narrow
    {180224ull, 2, 1, 1, 0},  // SENT/oneshot/fused
    {819200ull, 2, 1, 1, 1024},  // SENT/oneshot/fused/wide
    {1835008ull, 2, 2, 1, 0},  // SENT/twoshot/fused
    {7421952ull, 2, 2, 1, 1024},  // SENT/twoshot/fused/wide
    {51150848ull, 1, 2, 2, 0},  // LL128/twoshot/streamed
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
