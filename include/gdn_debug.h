/*
 * gdn_debug.h -- verification hooks, exported only by the test build of the library,
 * libgdn_test.so (the same sources compiled with GDN_TEST_HOOKS).  The product library libgdn.so
 * exports none of them: it has no switch that changes results and no fault hook.  The pages have
 * no counterpart to any of these calls.
 *
 * The chunk-wise prefill has two designs: the split path (a prep kernel for the state-independent
 * quantities of all chunks, then the state kernel) and the fused one-kernel path, which has two
 * builds of one data flow.  Mode 0 (the default and the product path) runs the split path when
 * the workspace holds it and the fused tensor-core build otherwise; mode 1 runs the fused build
 * with each MMA group replaced by a CUDA-core loop that reads the same swizzled shared-memory
 * operand tiles and writes the same tensor-memory accumulators; mode 2 runs the fused
 * tensor-core build whatever the workspace.  Comparing them isolates a fault to the tensor-core
 * descriptors, the fused data flow or the split data flow.  There is no counterpart on the pages.
 */
#ifndef GDN_DEBUG_H_
#define GDN_DEBUG_H_

#include "gdn.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Select the chunk-prefill build used by later gdn_chunk_prefill calls of libgdn_test.so in this
 * process: 0 = split path when the workspace allows, else fused (default); 1 = fused with CUDA-core
 * emulation of the MMAs; 2 = fused on the tensor cores.  A process-wide setting (an atomic store):
 * calls already issued keep the design they were issued with. */
GDN_API gdn_status gdn_debug_set_chunk_mode(int mode);

/* The mode last selected (0, 1 or 2). */
GDN_API int gdn_debug_get_chunk_mode(void);

/* One tensor-core tile, D = A * B^T: A [128][64] and B [n_cols][64] bf16 row-major (device),
 * D [128][n_cols] fp32 (device), n_cols 64 or 128.  The operands are staged in the same
 * 128-byte-swizzled K-major shared-memory layout and descriptors the chunk prefill uses.
 * *status (device, caller-zeroed) gets bit 0 if the bounded wait for the MMA ran out. */
GDN_API gdn_status gdn_debug_mma_probe(const gdn_bf16* A, const gdn_bf16* B, int n_cols, float* D,
                                       unsigned* status, void* stream);

/* The same tile with the operand placements of the split chunk prefill: flags bit 0 reads A
 * from tensor memory (two bf16 per 32-bit column, the even K index in the low half), bit 1 reads
 * B from an MN-major 128-byte-swizzled tile (128-byte rows of 64 N elements of one K index,
 * 64-element N blocks 8 KB apart).  Other flag bits are refused with GDN_ERR_INVALID_ARGUMENT. */
GDN_API gdn_status gdn_debug_mma_probe_ex(const gdn_bf16* A, const gdn_bf16* B, int n_cols, int flags, float* D,
                                          unsigned* status, void* stream);

/* Make a bounded in-kernel wait run out, to exercise the timeout path without a GPU fault.  Bit 0:
 * the binary16-state decode step (gdn_decode_step_fp16_state, staged form) arms its state-slice
 * barrier but issues no copy; bit 1: the split chunk prefill's state kernel does the same with the
 * first vector-block copy of each (sequence, head) item.  The wait on such a barrier runs out after
 * a short limit (4096 polls), the kernel raises the timeout bit of the device error word and
 * returns with nothing in flight (tensor memory released), and gdn_check_device_errors() then
 * returns GDN_ERR_TIMEOUT.  The outputs of the affected call are unspecified (the decode step has
 * already advanced the conv state).  0 restores normal operation.  Set on the current device.
 * Other bits: GDN_ERR_INVALID_ARGUMENT. */
GDN_API gdn_status gdn_debug_set_dropped_copy(unsigned which);

#ifdef __cplusplus
}
#endif

#endif /* GDN_DEBUG_H_ */
