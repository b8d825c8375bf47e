// kernels.h -- every kernel family's launch interface, for the C ABI layer
// (api.cu).  Each kernel translation unit includes only its own args_*.h, so
// that a change to one family's interface leaves the others' sources as they were.
#pragma once
#include "args_decode.h"
#include "args_merge.h"
#include "args_paged.h"
#include "args_prefill.h"
#include "args_verify.h"

namespace sinkattn {
// selftest.cu: one thread waits, with the library's bounded wait, on an mbarrier nothing completes.
cudaError_t wait_timeout_selftest_launch(unsigned* err, cudaStream_t stream);
}  // namespace sinkattn
