// profiler.hpp -- launch bracketing used by the kernel launchers (see
// profiler.cu).  Usage: prof::begin("name", stream); kernel<<<...>>>; prof::end(stream);
#pragma once

#include <cuda_runtime.h>

namespace nsa {
namespace prof {
bool enabled();
void begin(const char* name, cudaStream_t s);
void end(cudaStream_t s);
}  // namespace prof
}  // namespace nsa
