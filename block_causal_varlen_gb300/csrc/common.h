// Host-side helpers shared by the library's translation units.
#pragma once
#include <stdint.h>
#include <stddef.h>

#include "../../include/bd_attn.h"

namespace bd {

// Records `msg` (printf-style) as the calling thread's last error and returns `status`.
int32_t fail(int32_t status, const char* fmt, ...);

// Clears the calling thread's last error and returns BD_OK.
int32_t ok();

// Validated view of a host plan blob.
struct PlanView {
  const int32_t* w = nullptr;
  int32_t hdr(int i) const { return w[i]; }
  const int32_t* item(int i) const;
  const int32_t* seg(int i) const;
  const int32_t* fwd(int i) const;
  const int32_t* bwd(int i) const;
};

// Checks magic, version and internal offsets of a host plan blob.
int32_t view_plan(const void* plan_host, PlanView* out);

}  // namespace bd
