// Host-side plan object and call validation shared by plan.cpp and the CUDA entry points.
#pragma once

#include <string>
#include <vector>

#include "internal.h"

struct dattn_plan_s {
  dattn_problem prob;
  std::vector<int32_t> kv_len;
  std::vector<dattn::WorkItem> items;     // item order (group by group, chunk by chunk)
  std::vector<int32_t> item_cta;
  std::vector<uint8_t> blob;              // header + work list, copied by every run
  dattn_plan_info info;
  int32_t direct_items = 0;               // items that write O directly (no partial state)
};

namespace dattn {

// Collects every failed check (the rejection vector) before reporting.
struct Checker {
  dattn_status status = DATTN_OK;
  std::string reasons;
  void fail(dattn_status st, const std::string& why);
  dattn_status finish(const char* where);
};

void set_error(const std::string& s);
void check_problem(const dattn_problem* p, Checker& c);
bool same_problem(const dattn_problem& a, const dattn_problem& b);
int group_rows(const dattn_problem& p);

}  // namespace dattn
