/*
 * icp_timeline.h - measurement hook of the timeline build of libicp
 * (libicp_timeline.so, compiled with ICP_TIMELINE).  The ordinary library
 * does not export it.  Nothing on the FlashInfer msa_ops pages corresponds to
 * it: it exists to show where a scorer launch spends its time.
 *
 * In the timeline build every CTA of the decode scorer (icp_score, and the
 * fused icp_score_select) writes the global timer (ns) at these phases into
 * a fixed device array of 1024 CTAs x 24 slots:
 *    0  CTA entry
 *    1  set-up done (barriers, TMEM, per-request tile prefix sums)
 *    2  first index-K tile's TMA issued by the producer warp
 *    3  last index-K tile's TMA issued
 *    4  first tile's MMAs committed
 *    5  last tile's MMAs committed
 *    6-9  first tile finished by epilogue warp 0..3
 *   10  a tile finished by an epilogue warp (the last one written wins)
 *   11  CTA exit
 *   12  the producer's griddepcontrol.wait returned (early start only)
 *   13  the producer reached its first request (its queries' TMA issued)
 *   14  the producer's first block-table entries arrived
 *   15  thread 0 read its share of the request lengths
 *   16  the producer read its first request's length
 *   17  the first request's query slot was free
 *   18  the producer found its first tile in the prefix sums
 * Slots 19-23 hold per-CTA sums instead: the ns the producer waited for a
 * free ring stage (19); for the prefill scorer, the ns its MMA thread waited
 * for key tiles (20) and for an accumulator (21), and the ns its first
 * epilogue warp waited for a finished item (22); the number of request
 * segments (plan records) the CTA handled (23).  For the prefill scorer,
 * slot 4 / 5 are its first / last tile pair's MMAs committed and 6 / 10 its
 * first / last item finished by the first epilogue warp.
 * Slots a launch does not reach keep their previous contents.
 */
#ifndef ICP_TIMELINE_H
#define ICP_TIMELINE_H

#ifdef __cplusplus
extern "C" {
#endif

#define ICP_TIMELINE_CTAS 1024
#define ICP_TIMELINE_SLOTS 24

/*
 * Copies the stamps of CTAs 0 .. ctas-1 (ctas * 24 values, CTA-major) to the
 * HOST array dst, then, when clear is non-zero, zeroes the device array.
 * Synchronous (it waits for the device).  Returns 0, 1 for invalid arguments
 * (ctas outside [0, 1024], dst NULL), 2 when a CUDA call fails.
 */
int icp_timeline_read(unsigned long long *dst, int ctas, int clear);

#ifdef __cplusplus
}
#endif

#endif /* ICP_TIMELINE_H */
