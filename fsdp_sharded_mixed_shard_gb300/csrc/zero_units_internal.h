// zero_units_internal.h -- the unit plan object behind zero_units.h.
#ifndef ZERO_UNITS_INTERNAL_H
#define ZERO_UNITS_INTERNAL_H

#include <cstdint>
#include <vector>

#include "zero_units.h"

struct zero_unit_plan {
  zero_unit_plan_info info;
  std::vector<zero_unit> units;          // forward order
  std::vector<int32_t> slot_tensor;      // tensor ids unit by unit
  std::vector<int64_t> tensor_offset;    // per tensor, inside its gathered unit
};

#endif
