// Mutation driver for libdgt's host sources (packer, unpack, container),
// built with AddressSanitizer and UBSan by tests/test_host_sanitize.py.
// Each iteration packs a tensor (N(0, 0.02) weights, weights spread over
// 2^+-12 binades, or random bit patterns; format 1 or 2), flips bits in one
// of its arrays (or changes k), unpacks it, then writes a container, damages
// the file (truncation, bit flips, or a changed digit in the header), reads it
// and unpacks what it returns.  Every call must return a status; the
// sanitizers turn any out-of-bounds access or undefined behaviour into a
// non-zero exit.
// Usage: host_mutation_driver ITERATIONS WORKDIR SEED
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <random>
#include <string>
#include <vector>
#include <cmath>

#include "dgt.h"
int main(int argc, char **argv) {
    const int iters = argc > 1 ? atoi(argv[1]) : 200;
    std::mt19937_64 rng(argc > 3 ? strtoull(argv[3], nullptr, 10) : 12345);
    std::normal_distribution<float> nd(0.f, 0.02f);
    std::uniform_real_distribution<float> ud(-12.f, 12.f);
    std::vector<std::vector<uint16_t>> ws;
    const uint64_t R = 24, C = 1000;
    for (int kind = 0; kind < 3; kind++) {
        std::vector<uint16_t> w(R * C);
        for (auto &x : w) {
            float f = kind == 0 ? nd(rng) : (kind == 1 ? nd(rng) * std::exp2(ud(rng)) : 0.f);
            uint32_t u; std::memcpy(&u, &f, 4);
            x = kind == 2 ? (uint16_t)rng() : (uint16_t)(u >> 16);
        }
        ws.push_back(w);
    }
    std::vector<uint16_t> out(R * C);
    int errs = 0, oks = 0;
    for (int it = 0; it < iters; it++) {
        const auto &w = ws[it % 3];
        const int fmt = 1 + (it / 3) % 2;
        dgt_packed *p = nullptr;
        if (dgt_pack(w.data(), R, C, fmt, 2, &p) != DGT_OK) return 2;
        dgt_packed_view v;
        dgt_packed_get_view(p, &v);
        // flip bits in one of the arrays (the view points into the object)
        struct A { uint8_t *p; uint64_t n; } arrs[] = {
            {(uint8_t *)v.words, v.n_words * 4}, {(uint8_t *)v.blkq, v.n_blocks}, {(uint8_t *)v.grp, v.n_groups * 8},
            {(uint8_t *)v.payload, v.payload_bytes}, {(uint8_t *)v.tw, v.n_tiles}, {(uint8_t *)v.tesc, v.n_tiles},
            {(uint8_t *)v.esc1, v.n_esc1}, {(uint8_t *)v.grp1, v.n_groups1 * 12}};
        A a = arrs[rng() % 8];
        if (a.p && a.n)
            for (int f = 0, nf = 1 + rng() % 5; f < nf; f++) a.p[rng() % a.n] ^= (uint8_t)(1u << (rng() % 8));
        if (rng() % 4 == 0) v.rice_k = (int)(rng() % 9) - 1;
        (dgt_unpack(&v, out.data(), 2) == DGT_OK ? oks : errs)++;
        // the container: write, damage, read, unpack
        const char *nm = "t";
        std::string path = std::string(argv[2]) + "/c.dgt";
        if (dgt_write(path.c_str(), &p, &nm, 1) != DGT_OK) return 3;
        FILE *f = fopen(path.c_str(), "rb");
        std::vector<uint8_t> raw;
        int ch;
        while ((ch = fgetc(f)) != EOF) raw.push_back((uint8_t)ch);
        fclose(f);
        const int mode = rng() % 3;
        if (mode == 0) raw.resize(rng() % raw.size());
        else if (mode == 1) for (int k = 0; k < 4; k++) raw[rng() % raw.size()] ^= (uint8_t)(1u << (rng() % 8));
        else { uint64_t hl = 0; std::memcpy(&hl, raw.data(), 8); size_t at = 8 + rng() % hl; if (raw[at] >= '0' && raw[at] <= '9') raw[at] = '0' + rng() % 10; }
        f = fopen(path.c_str(), "wb");
        fwrite(raw.data(), 1, raw.size(), f);
        fclose(f);
        dgt_packed **ts = nullptr; char **ns = nullptr; int cnt = 0;
        if (dgt_read(path.c_str(), &ts, &ns, &cnt) == DGT_OK) {
            for (int i = 0; i < cnt; i++) {
                dgt_packed_view rv;
                dgt_packed_get_view(ts[i], &rv);
                std::vector<uint16_t> o2(rv.rows * rv.cols + 1);
                (dgt_unpack(&rv, o2.data(), 2) == DGT_OK ? oks : errs)++;
            }
            dgt_read_free(ts, ns, cnt);
        } else errs++;
        dgt_packed_free(p);
    }
    printf("ok %d err %d\n", oks, errs);
    return 0;
}
