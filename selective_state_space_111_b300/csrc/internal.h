// internal.h -- calls between the library's translation units (not part of
// the C ABI; hidden from the shared library's exported symbols).
#pragma once

#include <cstddef>

namespace ssm_internal {

// Chunk-state capture for the next forward calls made on this host thread:
// direction k (0 .. 3, in the form's own numbering: v1/v2 forward and
// backward branches 0 and 1, SS2D directions 0 .. 3) also stores its state
// before every kStateChunk-th walk step to hc[k], fp32 [B][D][ceil(L /
// kStateChunk)][16] (the layout the 16-state backward kernel reads).  Entries may be null; states
// beyond 16 are never captured.  Pass null to clear.
void set_chunk_state_capture(float *const *hc);

// The saved backward context set on this host thread (ssm_set_bwd_context),
// or null; *bytes receives its size.
void *bwd_context(size_t *bytes);

// Layout of a saved backward context of a sequence form with ndir
// directions (single: 1, v1 / v2: 2) and d_state <= 16: the pre-gate output
// [B][D][L] (esize bytes per element) at ypre, then direction k's
// chunk-start states at hc[k] (the capture layout above), each 256-byte
// aligned; total bytes.
struct CtxLayout {
    size_t ypre, hc[2], total;
};
CtxLayout ctx_layout(int ndir, unsigned esize, int B, int D, int L);

}  // namespace ssm_internal
