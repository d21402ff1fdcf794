// Ragged batches: segments of their own lengths laid end to end in one array,
// segment s holding elements offsets[s] .. offsets[s+1]-1, each fitted as its
// own row.  The paper ("Merge Hulls Without Copying Vertices", Section 7.7 and
// its conclusion) fits unequal segments either padded to a rectangle or laid
// end to end in one row with targets lifted per segment; here the offsets
// enter the library and each segment goes to the kernel made for its length.
//
// No host synchronisation: a classification kernel sorts the segments into
// lists on the device -- one per lane class (the smallest power of two L with
// 32 L >= length, L = 1 .. 256, rows of up to 8,192 elements) and one of long
// segments -- and every later kernel reads the list's count on the device.
// Grids are sized for the largest count the shape allows: a class of L >= 2
// holds segments longer than 16 L, so at most total / (16 L + 1) of them.
#include "../../include/iso.h"
#include "iso_internal.h"

#include <algorithm>

namespace isodev {

namespace {

constexpr int kClasses = 9;          // lane classes L = 1, 2, 4, ..., 256
constexpr int kLongList = kClasses;  // index of the long segments' counter

__host__ __device__ inline size_t align256r(size_t x) { return (x + 255) & ~size_t(255); }

// Largest number of segments of class k (k = kLongList: the long ones).
inline int64_t class_cap(int k, int64_t segments, int64_t total) {
    if (k == kLongList) return std::min<int64_t>(segments, total / (kRowMax + 1));
    if (k == 0) return std::min<int64_t>(segments, total);
    return std::min<int64_t>(segments, total / (16LL * (1LL << k) + 1));
}

// Lane class of a segment of n elements (1 <= n <= kRowMax).
inline __device__ int lane_class(int64_t n) {
    int k = 0;
    while ((32LL << k) < n) ++k;
    return k;
}

struct Lists {
    int32_t* list[kClasses + 1];          // per class, then the long segments
    int64_t cap[kClasses + 1];
    unsigned long long* count;            // [kClasses + 1], zeroed before the kernel
};

// Classification.  A segment whose offsets are out of order or out of range,
// or longer than max_len, gets ISO_ROW_BAD_SHAPE and is not fitted; an empty
// segment gets status 0.  The fitting kernels write the others' status.
__global__ void __launch_bounds__(256)
ragged_classify_kernel(const int64_t* __restrict__ off, int64_t segments, int64_t total,
                       int64_t max_len, Lists ls, uint32_t* __restrict__ row_status) {
    const int lane = threadIdx.x & 31;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t s = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; s < segments; s += stride) {
        const int64_t a = off[s], b = off[s + 1];
        int k = -1;
        uint32_t st = 0;
        if (a < 0 || b < a || b > total || b - a > max_len) st = ISO_ROW_BAD_SHAPE;
        else if (b > a) k = b - a > kRowMax ? kLongList : lane_class(b - a);
        // one atomic per class among the warp's active lanes
        const unsigned act = __activemask();
        const unsigned peers = __match_any_sync(act, k);
        const int leader = __ffs(peers) - 1;
        unsigned long long base = 0;
        if (k >= 0 && lane == leader) base = atomicAdd(&ls.count[k], (unsigned long long)__popc(peers));
        base = __shfl_sync(peers, base, leader);
        if (k >= 0) {
            const int64_t slot = (int64_t)base + __popc(peers & ((1u << lane) - 1u));
            if (slot < ls.cap[k]) ls.list[k][slot] = (int32_t)s;
            else st = ISO_ROW_BAD_SHAPE;   // more segments than the bound: overlapping offsets
        }
        if (row_status && (k < 0 || st)) row_status[s] = st;
    }
}

struct RaggedWs {
    Lists ls;
    void* long_ws;
    size_t bytes;
};

RaggedWs carve_ragged_ws(void* base, int64_t segments, int64_t total, int64_t max_len,
                         bool weighted) {
    RaggedWs r{};
    size_t off = 0;
    char* b = static_cast<char*>(base);
    auto take = [&](size_t bytes) -> void* {
        void* p = b ? (void*)(b + off) : nullptr;
        off += align256r(bytes);
        return p;
    };
    r.ls.count = (unsigned long long*)take(sizeof(unsigned long long) * (kClasses + 1));
    const int64_t lim = std::min<int64_t>(max_len, kRowMax);
    for (int k = 0; k <= kLongList; ++k) {
        const bool used = k == kLongList ? max_len > kRowMax : (k == 0 || (16LL << k) < lim);
        r.ls.cap[k] = used ? class_cap(k, segments, total) : 0;
        r.ls.list[k] = r.ls.cap[k] > 0 ? (int32_t*)take(sizeof(int32_t) * r.ls.cap[k]) : nullptr;
    }
    r.long_ws = nullptr;
    if (r.ls.cap[kLongList] > 0) {
        r.long_ws = b ? (void*)(b + off) : nullptr;
        off += long_ragged_workspace(r.ls.cap[kLongList], total, weighted);
    }
    r.bytes = off;
    return r;
}

}  // namespace

size_t ragged_workspace(int64_t segments, int64_t total, int64_t max_len, bool weighted) {
    return carve_ragged_ws(nullptr, segments, total, max_len, weighted).bytes;
}

template <class IO>
cudaError_t ragged_fit(const IO* y, const IO* w, const int64_t* off, int64_t segments,
                       int64_t total, int64_t max_len, int increasing, IO* out, uint8_t* blocks,
                       void* ws, uint32_t* row_status, cudaStream_t stream) {
    const RaggedWs r = carve_ragged_ws(ws, segments, total, max_len, w != nullptr);
    cudaError_t err = cudaMemsetAsync(r.ls.count, 0, sizeof(unsigned long long) * (kClasses + 1),
                                      stream);
    if (err != cudaSuccess) return err;
    const int64_t grid = std::min<int64_t>((segments + 255) / 256, kRaggedCtas);
    ragged_classify_kernel<<<(unsigned)grid, 256, 0, stream>>>(off, segments, total, max_len,
                                                               r.ls, row_status);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    prof_mark(stream, "ragged_classify");
    for (int k = 0; k < kClasses; ++k) {
        if (r.ls.cap[k] == 0) continue;
        err = rows_fit_ragged<IO>(y, w, off, r.ls.list[k], r.ls.count + k, r.ls.cap[k], 1 << k,
                              increasing, out, blocks, row_status, stream);
        if (err != cudaSuccess) return err;
    }
    if (r.ls.cap[kLongList] > 0)
        return long_fit_ragged<IO>(y, w, off, r.ls.list[kLongList], r.ls.count + kLongList,
                                   r.ls.cap[kLongList], total, increasing, out, blocks, r.long_ws,
                                   row_status, stream);
    return cudaSuccess;
}

template cudaError_t ragged_fit<float>(const float*, const float*, const int64_t*, int64_t,
                                       int64_t, int64_t, int, float*, uint8_t*, void*, uint32_t*,
                                       cudaStream_t);
template cudaError_t ragged_fit<double>(const double*, const double*, const int64_t*, int64_t,
                                        int64_t, int64_t, int, double*, uint8_t*, void*,
                                        uint32_t*, cudaStream_t);

}  // namespace isodev
