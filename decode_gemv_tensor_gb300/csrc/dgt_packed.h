// dgt_packed.h -- the library-owned host object behind dgt_packed*.
#pragma once
#include <memory>
#include <new>
#include <type_traits>
#include <utility>
#include <vector>

#include "../../include/dgt.h"

// An allocator whose construct() default-initialises: resize() leaves new
// elements of a trivial type uninitialised, so a large array is first touched
// by the threads (or the file read) that fill it instead of by a serial
// zero fill.
template <class T>
struct DefaultInitAlloc : std::allocator<T> {
    template <class U>
    struct rebind {
        using other = DefaultInitAlloc<U>;
    };
    DefaultInitAlloc() = default;
    template <class U>
    DefaultInitAlloc(const DefaultInitAlloc<U> &) noexcept {}
    template <class U>
    void construct(U *p) noexcept(std::is_nothrow_default_constructible<U>::value) {
        ::new ((void *)p) U;
    }
    template <class U, class... Args>
    void construct(U *p, Args &&...args) {
        ::new ((void *)p) U(std::forward<Args>(args)...);
    }
};

struct dgt_packed {
    dgt_packed_view v;
    std::vector<uint8_t, DefaultInitAlloc<uint8_t>> sm;   // every byte written by its producer
    std::vector<uint8_t> blkq, payload, tw, tesc, esc1;
    std::vector<uint32_t> words, grp, grp1;
    // Point the view at the vectors (after any of them changed size).
    void refresh() {
        v.sm = sm.data();
        v.words = words.data();
        v.n_words = words.size();
        v.blkq = blkq.data();
        v.n_blocks = blkq.size();
        v.grp = grp.data();
        v.n_groups = grp.size() / 2;
        v.payload = payload.data();
        v.payload_bytes = payload.size();
        v.tw = tw.data();
        v.tesc = tesc.data();
        v.n_tiles = tw.size();
        v.esc1 = esc1.data();
        v.n_esc1 = esc1.size();
        v.grp1 = grp1.data();
        v.n_groups1 = grp1.size() / 3;
    }
};
