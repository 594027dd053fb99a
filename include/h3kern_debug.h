/*
 * h3kern test hooks.  Not part of the production interface; the page
 * material has no counterpart for these -- they exist so the bounded-wait
 * failure path of the attention kernel can be exercised without faulting,
 * trapping or hanging a GPU.
 */
#ifndef H3KERN_DEBUG_H
#define H3KERN_DEBUG_H

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Arms a one-shot fault for the next h3_attention launch (from any thread).
 *   fault = 0  disarm
 *   fault = 1  the TMA producer of every CTA skips loading K/V tile 1, so
 *              the MMA issuer's bounded wait runs out (about 2 s of wall
 *              clock); the kernel sets H3_STATUS_TIMEOUT_MMA (and possibly
 *              other timeout / abort bits) in the status word, drains its
 *              in-flight copies and MMAs, frees TMEM and returns.  The
 *              output is then undefined; h3_status_word() reports the bits.
 *              Needs a segment with at least 2 KV tiles (> 128 valid keys).
 * Returns H3_OK, or H3_ERR_ARG for an unknown fault.
 */
int h3_debug_fault_next_attention(int fault);

#ifdef __cplusplus
}
#endif

#endif /* H3KERN_DEBUG_H */
