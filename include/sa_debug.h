/*
 * sa_debug.h -- test entry point of the SA_DEBUG build of the library
 * (libsa_gb300_debug.so; build with build.build(debug=True)).  The release
 * library does not export it.  The pages describe no such step: it is a
 * debugging aid of this implementation.
 *
 * In the SA_DEBUG build every tensor-core kernel checks each work description
 * it reads before touching memory through it: a band item's residue class
 * must lie among the problem's classes and in the launch's window of tensor
 * maps, its head in [0, B*H), its query tile and each key-tile range it lists
 * inside the class; a global-row item's head, key chunk and tile of global
 * rows inside the problem.  An item that fails is skipped by every role of the
 * CTA (no tile is loaded, no output row written) and the device error word
 * gets the bit that sa_sync_status() reports as SA_ERR_CUDA ("a kernel failed
 * a device-side check").  The arithmetic is that of the release build.
 */
#ifndef SA_DEBUG_H_
#define SA_DEBUG_H_

#include "sa.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Runs the band-item range check of the SA_DEBUG kernels by itself, in a
 * kernel of its own, over a list of work items, and counts the items that
 * fail it.  Nothing else runs, so a list with bad entries is safe to check.
 *
 *  items     host array of n_items band items, each eight int32 in the order
 *            {head (b*H + h), residue-class slot, first query tile, flags,
 *             first key tile of query tile 0, of query tile 1,
 *             last key tile of query tile 0, of query tile 1}
 *            (a query tile whose last key tile is below its first is empty).
 *  slots     host array of n_slots residue classes, four int32 each
 *            {dilation d, residue r, length ceil((N - r) / d), unused}.
 *  slot_base first class of the launch window (its tensor maps cover classes
 *            slot_base .. slot_base + 15).
 *  BH        batch x heads.
 *  n_bad     out: the number of items that fail the check.
 *
 * Host arrays are read during the call only.  The call is synchronous (it
 * allocates, copies, runs and frees on the legacy default stream).  Returns
 * SA_ERR_INVALID_ARG for a null pointer or a negative count, SA_ERR_CUDA if
 * a CUDA call fails.
 */
sa_status sa_debug_check_band_items(const void *items, int n_items, const void *slots,
                                    int n_slots, int slot_base, int BH, int *n_bad);

#ifdef __cplusplus
}
#endif

#endif /* SA_DEBUG_H_ */
