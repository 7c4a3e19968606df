// Causal varlen paged prefill (tcgen05 / TMEM / TMA). Not built yet: the launcher
// reports PGQA_EUNSUPPORTED so that callers fail loudly.
#include "host.h"

namespace pgqa {

pgqa_status_t launch_paged_prefill(const PrefillArgs& a) {
  (void)a;
  return PGQA_EUNSUPPORTED;
}

}  // namespace pgqa
