// Internal interface between the plan code (cs_chain.cu) and the tuning table
// (cs_tune.cpp).  Not part of the C ABI.
#pragma once

#include "../../include/cs_chain.h"

// Records a status and its message as the thread's last error; returns s.
cs_status cs_fail(cs_status s, const char* fmt, ...);

// Looks up the tuning-table entry for a desc run on num_sms SMs.  Returns the
// entry's index, or -1 when the table is not consulted (desc->tuned < 0, or no
// field it may fill is auto) or holds no entry for this shape.  On a match,
// *out is *in with the entry's policy (when in->policy is CS_SYNC_AUTO) and
// tile_m / tile_n / split_k / group_m (when all four are auto in *in) applied,
// and its Stream-K tail (sk_tiles / sk_units) when those are auto too.
int cs_tune_apply(const cs_chain_desc* in, int num_sms, cs_chain_desc* out);
