// Internal interface between the C ABI (clsample.cu) and the persistent streaming
// sampler (stream.cu).  Not part of the public header.
#pragma once

#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "clsample.h"

namespace clsample_stream {

// True when the streaming sampler produces every output the call asks for: all calls
// except those with requested-id logprobs, top-N logprobs or the joint top-k/top-p mode
// (those run on the slice-resident kernel).
bool serves(const clsample_args_t* a);

// Rows one launch takes; larger batches are split into launches of at most this many.
constexpr int kMaxRows = 1024;

// Bytes of device scratch for batches of up to max_batch rows over `vocab` tokens.
size_t scratch_bytes(int max_batch, int vocab);

// Once per device: sets the kernel's shared-memory limit and returns in *grid the number
// of CTAs that are resident at once (the persistent grid).
int setup(int dev, int* grid);

// Enqueues one call on `st` (one kernel launch per kMaxRows rows).  `scratch` holds
// scratch_bytes(max_batch, V) bytes that were zero when first used; every launch leaves
// its counters at zero again and advances the scratch's launch epoch (kept on the
// device, so a launch replayed from a CUDA graph takes a fresh one).  Arguments are
// validated by the caller.
int launch(const clsample_args_t* a, unsigned char* scratch, int max_batch, int grid, cudaStream_t st);

}  // namespace clsample_stream
