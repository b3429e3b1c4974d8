// Host helpers shared by the two C-ABI translation units (abi.cu, and
// noalloc.cu for the allocation-free entry point), so that both build the
// kernels' parameter blocks the same way.
#pragma once

#include "kernels.h"
#include "moe.h"

namespace moe_abi {

// Largest byte offset + size of the nine sub-tensors of one expert blob.
size_t blob_extent(const moe_layer_weights &w);

// The kernels' view of a layer description (pointers, blob layout, options).
moe::LayerPtrs layer_ptrs(const moe_layer_weights &w);

// Host-side validation of a layer description (MOE_OK or an error code).
int check_weights(const moe_layer_weights *w);

// Whether the fused single-token kernel can run this shape on a device with
// n_sm multiprocessors (one router row per block, one block per SM).
bool decode_fused_supported(const moe_dims &d, int n_sm);

}  // namespace moe_abi
