// The draft stage behind both of its entry points, spec_draft_sample
// (caller workspace) and spec_draft_sample_static (library scratch) (internal
// header).
#pragma once

#include "common.cuh"
#include "spec.h"

namespace spec {

// Argument checks shared by both entry points (the workspace is not checked).
int check_draft_args(const spec_draft_args* a);

// True when the fused tensor-core kernels take the draft; *sms is the device's
// SM count then.
bool draft_tc_ok(const spec_draft_args& a, int* sms);

// Every launch of one draft call: the counters memset, the draft steps (fused
// when tc_sms > 0, for a device of tc_sms SMs; generic otherwise), the
// optional full distributions and the confidence head.  `partials` and
// `counters` ([R] counters then [gamma, R] race bounds) are scratch sized for
// the path taken.
int run_draft(const spec_draft_args& a, uint64_t seed, Partial* partials, unsigned* counters,
              int tc_sms, cudaStream_t stream);

}  // namespace spec
