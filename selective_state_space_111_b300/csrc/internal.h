// internal.h -- calls between the library's translation units (not part of
// the C ABI; hidden from the shared library's exported symbols).
#pragma once

namespace ssm_internal {

// Chunk-state capture for the next forward calls made on this host thread:
// direction k (0 .. 3, in the form's own numbering: v1/v2 forward and
// backward branches 0 and 1, SS2D directions 0 .. 3) also stores its state
// before every kStateChunk-th walk step to hc[k], fp32 [B][D][ceil(L /
// kStateChunk)][16] (the layout the 16-state backward kernel reads).  Entries may be null; states
// beyond 16 are never captured.  Pass null to clear.
void set_chunk_state_capture(float *const *hc);

}  // namespace ssm_internal
