// dgt_packed.h -- the library-owned host object behind dgt_packed*.
#pragma once
#include <vector>

#include "../../include/dgt.h"

struct dgt_packed {
    dgt_packed_view v;
    std::vector<uint8_t> sm, blkq, payload, tw, tesc, esc1;
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
