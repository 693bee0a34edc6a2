// ce_span.cuh -- splitting a run of row elements at 16-byte boundaries.
//
// A row of V elements of type T starts wherever its strides put it: rows of
// a vocabulary that is not a multiple of 16 / sizeof(T) (50257, 100277, ...)
// or padded views start off a 16-byte boundary.  The streaming kernels that
// take such rows read the elements [e0, e1) as
//   head: the elements before the first 16-byte boundary (< 16 / sizeof(T)),
//   body: whole 16-byte vectors,
//   tail: what follows the last whole vector (< 16 / sizeof(T)),
// so every access stays inside [e0, e1) and the bulk of the run moves in
// 16-byte loads and stores.  The row must sit on a multiple of sizeof(T)
// (the entry points refuse logits that do not), so the head is a whole
// number of elements.  On an aligned run the head and tail are empty.
#pragma once

#include <cstdint>

namespace gbce {

struct Span16 {
    int64_t h1;  // first element of the body (end of the head)
    int64_t nv;  // whole 16-byte vectors in the body
    int64_t t0;  // first element of the tail
};

template <int ES>
__device__ __forceinline__ Span16 span16(const void* row, int64_t e0, int64_t e1) {
    constexpr int VEC = 16 / ES;
    const uint32_t mis = (uint32_t)(reinterpret_cast<uintptr_t>(row) + (uintptr_t)(e0 * ES)) & 15u;
    const int64_t len = e1 > e0 ? e1 - e0 : 0;  // a chunk past the row's end is empty
    int64_t head = (int64_t)(((16u - mis) & 15u) / ES);
    if (head > len) head = len;
    Span16 s;
    s.h1 = e0 + head;
    s.nv = (len - head) / VEC;
    s.t0 = s.h1 + s.nv * VEC;
    return s;
}

// The element that thread t takes among the head and tail of [e0, e1)
// (head first), or -1: together they hold at most 2 (16 / ES - 1) elements,
// so one pass of any CTA of 32 or more threads covers them.
__device__ __forceinline__ int64_t span16_edge(const Span16& s, int64_t e0, int64_t e1, int t) {
    const int64_t head = s.h1 - e0;
    const int64_t e = t < head ? e0 + t : s.t0 + (t - head);
    return e < e1 ? e : -1;
}

}  // namespace gbce
