/*
 * zero_internal.h -- host-side plan representation shared by the planner
 * (plan.cpp) and the launch layer (zero_kernels.cu). Not part of the ABI.
 */
#ifndef ZERO_INTERNAL_H
#define ZERO_INTERNAL_H

#include <cstdint>
#include <vector>

#include "zero.h"

struct zero_plan {
  zero_plan_info info;
  std::vector<int64_t> offsets;       // per tensor
  std::vector<zero_segment> segs;     // ordered by lo
  std::vector<int64_t> seg_tile0;     // first norm tile of each segment (global numbering)
  std::vector<int64_t> seg_tiles;     // tiles in each segment
  std::vector<int32_t> rank_seg0;     // first segment of each rank, plus a sentinel
};

namespace zero_detail {
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
// norm finish: share records per owner that the workspace holds after the
// tile records (one 16-byte record each)
constexpr int kNormOwnerBlocks = 16;
}  // namespace zero_detail

#endif
