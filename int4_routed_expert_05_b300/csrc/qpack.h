// qpack.h -- the expert container's reader as the rest of the library uses it (see qpack.cpp).
#pragma once
#include <cstdint>

#include "moe.h"

namespace moe {
// Message for moe_last_error() (defined with the other entry points).
void set_last_error(const char* msg);

namespace qp {
// Reads blobs (layer[i], expert[i]) of the container into dst[i] (stride bytes each; 4096-byte
// aligned when the container was opened for direct reads), in parallel on the container's reader
// threads; returns when all are done: 0, or the errno of a failed read.
int read_many(moe_qpack* q, int n, const int32_t* layer, const int32_t* expert, void* const* dst);
uint64_t stride(const moe_qpack* q);
int n_layers(const moe_qpack* q);
const moe_shape& shape(const moe_qpack* q);
}  // namespace qp
}  // namespace moe
