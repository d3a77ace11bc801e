// store.cpp -- the expert container file: every routed expert of every layer
// as one fixed-stride blob, so fetching an expert is one positioned read.
//
// Swiftlet keeps its routed experts on the SSD in a container of fixed-stride
// blobs and reads each with a single pread, without mmap and without page-
// cache thrash (article section 2 "Fixed-stride pread reads"; README "How it
// works": the repacked .qpack container).  The pages do not give the
// container's layout; this library's is:
//
//   offset 0     header, 4096 bytes, little-endian (struct FileHeader below,
//                zero-padded)
//   offset 4096  blob (layer l, expert e) at 4096 + (l * n_experts + e) * stride
//
// The stride is the blob stride of moe_blob_stride (a multiple of 4096), so
// every blob starts and ends on a 4096-byte boundary and O_DIRECT reads of a
// blob need no bounce buffer.
#ifndef _GNU_SOURCE
#define _GNU_SOURCE  // O_DIRECT
#endif
#include <errno.h>
#include <fcntl.h>
#include <sys/stat.h>
#include <unistd.h>

#include <cstring>

#include "moe_internal.h"
#include "store.h"

namespace moe {
namespace {

constexpr char kMagic[8] = {'M', 'O', 'E', 'X', 'P', 'R', 'T', '1'};
constexpr uint32_t kVersion = 1;
constexpr uint64_t kHeaderBytes = 4096;

struct FileHeader {
    char magic[8];
    uint32_t version;
    uint32_t n_layers, n_experts, hidden, inter, bits, group_size;
    uint32_t pad;
    uint64_t stride;
    uint64_t data_offset;
};
static_assert(sizeof(FileHeader) == 56, "container header layout (bytes 0..55 of the 4096-byte header)");

// Byte order: the header is written field by field as little-endian.
void put32(uint8_t* p, uint32_t v) {
    for (int i = 0; i < 4; ++i) p[i] = (uint8_t)(v >> (8 * i));
}
void put64(uint8_t* p, uint64_t v) {
    for (int i = 0; i < 8; ++i) p[i] = (uint8_t)(v >> (8 * i));
}
uint32_t get32(const uint8_t* p) {
    uint32_t v = 0;
    for (int i = 0; i < 4; ++i) v |= (uint32_t)p[i] << (8 * i);
    return v;
}
uint64_t get64(const uint8_t* p) {
    uint64_t v = 0;
    for (int i = 0; i < 8; ++i) v |= (uint64_t)p[i] << (8 * i);
    return v;
}

void encode(const StoreShape& s, uint8_t* out) {
    std::memset(out, 0, kHeaderBytes);
    std::memcpy(out, kMagic, 8);
    put32(out + 8, kVersion);
    put32(out + 12, (uint32_t)s.n_layers);
    put32(out + 16, (uint32_t)s.n_experts);
    put32(out + 20, (uint32_t)s.hidden);
    put32(out + 24, (uint32_t)s.inter);
    put32(out + 28, (uint32_t)s.bits);
    put32(out + 32, 64u);
    put64(out + 40, s.stride);
    put64(out + 48, kHeaderBytes);
}

int decode(const uint8_t* in, StoreShape& s) {
    if (std::memcmp(in, kMagic, 8) != 0 || get32(in + 8) != kVersion) return MOE_EIO;
    s.n_layers = (int32_t)get32(in + 12);
    s.n_experts = (int32_t)get32(in + 16);
    s.hidden = (int32_t)get32(in + 20);
    s.inter = (int32_t)get32(in + 24);
    s.bits = (int32_t)get32(in + 28);
    if (get32(in + 32) != 64u || get64(in + 48) != kHeaderBytes) return MOE_EIO;
    s.stride = get64(in + 40);
    return MOE_OK;
}

// Whole-buffer positioned I/O: loops over short transfers and EINTR.
int pread_all(int fd, void* buf, size_t n, uint64_t off) {
    uint8_t* p = static_cast<uint8_t*>(buf);
    while (n > 0) {
        const ssize_t r = ::pread(fd, p, n, (off_t)off);
        if (r < 0) {
            if (errno == EINTR) continue;
            return MOE_EIO;
        }
        if (r == 0) return MOE_EIO;  // past the end of the file: a truncated container
        p += r, n -= (size_t)r, off += (uint64_t)r;
    }
    return MOE_OK;
}

int pwrite_all(int fd, const void* buf, size_t n, uint64_t off) {
    const uint8_t* p = static_cast<const uint8_t*>(buf);
    while (n > 0) {
        const ssize_t r = ::pwrite(fd, p, n, (off_t)off);
        if (r < 0) {
            if (errno == EINTR) continue;
            return MOE_EIO;
        }
        p += r, n -= (size_t)r, off += (uint64_t)r;
    }
    return MOE_OK;
}

bool valid_shape(const StoreShape& s) {
    return s.n_layers >= 1 && s.n_experts >= 1 && s.hidden > 0 && s.inter > 0 && (s.bits == 4 || s.bits == 8) &&
           s.stride > 0 && s.stride % 4096 == 0;
}

}  // namespace

uint64_t store_blob_offset(const StoreShape& s, int layer, int expert) {
    return kHeaderBytes + ((uint64_t)layer * (uint64_t)s.n_experts + (uint64_t)expert) * s.stride;
}

int store_create(const char* path, const StoreShape& s) {
    if (!path || !valid_shape(s)) return MOE_EINVAL;
    const int fd = ::open(path, O_WRONLY | O_CREAT | O_TRUNC | O_CLOEXEC, 0644);
    if (fd < 0) return MOE_EIO;
    uint8_t hdr[kHeaderBytes];
    encode(s, hdr);
    int rc = pwrite_all(fd, hdr, kHeaderBytes, 0);
    const uint64_t total = store_blob_offset(s, s.n_layers, 0);
    if (rc == MOE_OK && ::ftruncate(fd, (off_t)total) != 0) rc = MOE_EIO;
    if (::close(fd) != 0 && rc == MOE_OK) rc = MOE_EIO;
    return rc;
}

int store_open(const char* path, bool direct, StoreFile& f) {
    f = StoreFile{};
    if (!path) return MOE_EINVAL;
    // header and length through a buffered descriptor
    int fd = ::open(path, O_RDONLY | O_CLOEXEC);
    if (fd < 0) return MOE_EIO;
    uint8_t hdr[kHeaderBytes];
    int rc = pread_all(fd, hdr, kHeaderBytes, 0);
    if (rc == MOE_OK) rc = decode(hdr, f.shape);
    if (rc == MOE_OK && !valid_shape(f.shape)) rc = MOE_EIO;
    struct stat st {};
    if (rc == MOE_OK && (::fstat(fd, &st) != 0 ||
                         (uint64_t)st.st_size < store_blob_offset(f.shape, f.shape.n_layers, 0)))
        rc = MOE_EIO;  // shorter than its header says
    if (rc == MOE_OK && direct) {
        const int dfd = ::open(path, O_RDONLY | O_CLOEXEC | O_DIRECT);
        if (dfd >= 0) {
            ::close(fd);
            fd = dfd;
        } else {
            direct = false;  // no direct I/O on this file system: read through the page cache
        }
    }
    if (rc != MOE_OK) {
        ::close(fd);
        f = StoreFile{};
        return rc;
    }
    f.fd = fd;
    f.direct = direct;
    return MOE_OK;
}

void store_close(StoreFile& f) {
    if (f.fd >= 0) ::close(f.fd);
    f = StoreFile{};
}

int store_write_layer(const char* path, int layer, const void* blobs, size_t stride) {
    if (!path || !blobs) return MOE_EINVAL;
    StoreFile f;
    int rc = store_open(path, false, f);
    if (rc) return rc;
    const StoreShape s = f.shape;
    store_close(f);
    if (layer < 0 || layer >= s.n_layers || stride != s.stride) return MOE_EINVAL;
    const int fd = ::open(path, O_WRONLY | O_CLOEXEC);
    if (fd < 0) return MOE_EIO;
    rc = pwrite_all(fd, blobs, (size_t)s.n_experts * s.stride, store_blob_offset(s, layer, 0));
    if (::close(fd) != 0 && rc == MOE_OK) rc = MOE_EIO;
    return rc;
}

int store_read_blob(const StoreFile& f, int layer, int expert, void* dst) {
    if (f.fd < 0 || layer < 0 || layer >= f.shape.n_layers || expert < 0 || expert >= f.shape.n_experts || !dst)
        return MOE_EINVAL;
    if (f.direct && (reinterpret_cast<uintptr_t>(dst) % 4096) != 0) return MOE_EINVAL;
    return pread_all(f.fd, dst, f.shape.stride, store_blob_offset(f.shape, layer, expert));
}

}  // namespace moe

// ---------------------------------------------------------------------------
// C ABI
// ---------------------------------------------------------------------------
extern "C" int moe_store_create(const char* path, int32_t n_layers, int32_t n_experts, int32_t hidden, int32_t inter,
                                int32_t bits) {
    moe::StoreShape s{};
    s.n_layers = n_layers, s.n_experts = n_experts, s.hidden = hidden, s.inter = inter, s.bits = bits;
    s.stride = moe_blob_stride(hidden, inter, bits);
    if (s.stride == 0) return MOE_EINVAL;
    return moe::store_create(path, s);
}

extern "C" int moe_store_write_layer(const char* path, int32_t layer, const void* blobs_host, size_t stride) {
    return moe::store_write_layer(path, layer, blobs_host, stride);
}

extern "C" int moe_store_info(const char* path, int32_t* shape_out, uint64_t* stride_out) {
    if (!path || !shape_out || !stride_out) return MOE_EINVAL;
    moe::StoreFile f;
    const int rc = moe::store_open(path, false, f);
    if (rc) return rc;
    shape_out[0] = f.shape.n_layers, shape_out[1] = f.shape.n_experts, shape_out[2] = f.shape.hidden;
    shape_out[3] = f.shape.inter, shape_out[4] = f.shape.bits;
    *stride_out = f.shape.stride;
    moe::store_close(f);
    return MOE_OK;
}

extern "C" int moe_store_read(const char* path, int32_t layer, int32_t expert, void* dst_host, size_t cap) {
    if (!path || !dst_host) return MOE_EINVAL;
    moe::StoreFile f;
    int rc = moe::store_open(path, false, f);
    if (rc) return rc;
    rc = cap < f.shape.stride ? MOE_EINVAL : moe::store_read_blob(f, layer, expert, dst_host);
    moe::store_close(f);
    return rc;
}
