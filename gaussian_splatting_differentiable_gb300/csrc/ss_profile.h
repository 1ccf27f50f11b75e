// Per-kernel CUDA-event timing scope (see ss_profile.cu).
#pragma once

#include <cuda_runtime.h>

namespace ss {

bool profile_on();

// Records an event on `s` at construction and at destruction when profiling
// is on; wrap exactly one kernel launch.
class ProfScope {
  public:
    ProfScope(const char *name, cudaStream_t s);
    ~ProfScope();
    ProfScope(const ProfScope &) = delete;
    ProfScope &operator=(const ProfScope &) = delete;

  private:
    const char *name_;
    cudaStream_t s_;
    cudaEvent_t a_;
};

}  // namespace ss

// Launch one kernel inside a profiling scope named `name`.
#define SS_LAUNCH(name, stream, ...)          \
    do {                                      \
        ::ss::ProfScope ss_ps_(name, stream); \
        __VA_ARGS__;                          \
    } while (0)
