// store.h -- the expert container file (fixed-stride blobs, positioned reads).
#pragma once

#include <stddef.h>
#include <stdint.h>

namespace moe {

struct StoreShape {
    int32_t n_layers = 0, n_experts = 0, hidden = 0, inter = 0, bits = 0;
    uint64_t stride = 0;
};

struct StoreFile {
    int fd = -1;          // blob reads (O_DIRECT when `direct`)
    bool direct = false;  // direct reads want 4096-aligned destinations
    StoreShape shape;
};

uint64_t store_blob_offset(const StoreShape& s, int layer, int expert);
// Creates (or truncates) the container: header, then room for every blob.
int store_create(const char* path, const StoreShape& s);
// Opens a container and checks its header and length; `direct` asks for
// O_DIRECT blob reads and falls back to buffered ones where the file system
// has none.
int store_open(const char* path, bool direct, StoreFile& f);
void store_close(StoreFile& f);
// One blob (stride bytes) into dst: a single positioned read, repeated only
// over short transfers.
int store_read_blob(const StoreFile& f, int layer, int expert, void* dst);
// All blobs of one layer from a host buffer [n_experts][stride].
int store_write_layer(const char* path, int layer, const void* blobs, size_t stride);

}  // namespace moe
