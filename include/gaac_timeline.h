/*
 * Per-CTA timeline of the decode-attention kernel: a diagnostic of the
 * library's own launch behaviour (how long each CTA's split takes, how long
 * each block's copy is in flight, how long the split merge runs), not part of
 * the GAAC method.  Only a library built with -DGAAC_TIMELINE exports it
 * (lossless_compressed_kv_gaac_gb300/build.py, timeline=True: libgaac_timeline.so);
 * the default library has no instrumentation and no such symbol.
 *
 * Every attention launch of a timeline build overwrites, for CTA id
 * x + X * (y + Y * z) < n_ctas (grid (X, Y, Z) = (split, kv-head, sequence)),
 * one record of %globaltimer nanoseconds:
 *   u64 start, split_end, exit, merged;   (merged: 0 unless this CTA merged)
 *   u64 issue[n_blocks], arrive[n_blocks], land[n_blocks], release[n_blocks];
 * for the split's blocks j < n_blocks (copy issued; the first warp of the
 * block's group starts waiting for it, and passes the wait; the last warp of
 * the group is done with the stage).
 * gaac_timeline_fetch copies min(bytes, n_ctas * cta_bytes) bytes of the
 * records to host memory (host_dst may be NULL to query the sizes only).
 * Returns GAAC_OK or GAAC_ECUDA.
 */
#pragma once
#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

int gaac_timeline_fetch(void* host_dst, size_t bytes, size_t* cta_bytes, int* n_ctas, int* n_blocks);

#ifdef __cplusplus
}
#endif
