// Host-side helpers shared by the translation units of libspecverify.so.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace sv {
int sm_count();                    // SMs of the current device
void prof_begin(cudaStream_t s);   // profiling hook around the dominant kernel
void prof_end(cudaStream_t s);
void set_launches(int n);          // kernels launched by the last call (this thread)
void counter_region(int B, int rows, int V, size_t *offset, size_t *bytes);  // per-request counters
}  // namespace sv
