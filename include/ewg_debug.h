/*
 * Test hooks of the bounds-checking build (libewg_debug.so, compiled with EWG_DEBUG).
 * The ordinary library does not export them.
 */
#ifndef EWG_DEBUG_H
#define EWG_DEBUG_H

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Runs the listing's decoupled look-back once, from tile `tile`, on one warp of one CTA,
 * over `words` (device memory, tile + 1 uint32 words, one per tile; the caller owns it):
 * word j holds 0 (tile j has not published), (1 << 30) | count (its own count) or
 * (2 << 30) | count (the sum over it and every tile before it).  The probe sums the
 * predecessors' counts back to the first word that holds a sum, re-polling unpublished
 * words at most poll_limit times, then publishes word[tile] = (2 << 30) | (sum + 1).
 * Writes out[0] = 1 if it completed and 0 if it gave up on an unpublished word, and
 * out[1] = the sum it found (device memory, two ints).  Stream-ordered on `stream`.
 * Returns EWG_ERR_INVALID for null pointers, tile < 1 or poll_limit < 1, EWG_ERR_CUDA if
 * the launch fails, EWG_OK otherwise.  This is how a predecessor that never publishes is
 * injected from the host: the look-back must end on its own and report it.
 */
int ewg_debug_lookback_probe(void* words, int tile, int poll_limit, int* out, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* EWG_DEBUG_H */
