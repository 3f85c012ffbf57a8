// RAII bracket of one kernel launch for the optional per-kernel timing.
#pragma once
#include <cuda_runtime.h>

namespace rpa {
bool prof_enabled();  // per-kernel timing on: launches are bracketed, so nothing may overlap

class ProfScope {
   public:
    ProfScope(const char* name, cudaStream_t s);
    ~ProfScope();

   private:
    const char* name_;
    cudaStream_t stream_;
    void* a_;
    void* b_;
};
}  // namespace rpa
