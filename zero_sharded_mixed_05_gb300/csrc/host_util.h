// host_util.h -- host-side helpers shared by the library's translation units.
#pragma once

#include "zero_opt.h"
#include "zero_opt_internal.h"

namespace zo {

// Record a formatted message for zero_opt_last_error() and return `s`.
zero_status fail(zero_status s, const char* fmt, ...);

// Shard of `rank` for numel elements over world ranks: begin = rank*S, the
// number of real (non-padding) elements, and S.
void shard_range(int64_t numel, int32_t world, int32_t rank, int64_t* begin,
                 int64_t* real_len, int64_t* shard_len);

// EINVAL (with a message) unless every field of the configuration is valid.
zero_status check_config(const zero_opt_config* c);

// The configuration's hyperparameters as the decision takes them, with the
// gradient divisor D.
Hyper hyper_of(const zero_opt_config& c, double divisor);

}  // namespace zo
