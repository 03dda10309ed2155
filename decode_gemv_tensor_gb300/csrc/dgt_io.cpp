// dgt_io.cpp -- the packed-checkpoint container.
//
// The model cards of the packed models (Hugging Face pages for the 3B, 12B and
// 26B-A4B checkpoints, "Requirements and limits") store the packed bytes as
// uint8 tensors next to header metadata that records the format.  This file
// writes and reads that container as a safetensors file: a little-endian u64
// header length, a JSON header (dtype "U8", shape, data_offsets per array, and
// a "__metadata__" string map), then the concatenated array bytes.
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <memory>
#include <new>
#include <string>
#include <vector>

#include <unistd.h>

#include "../../include/dgt.h"
#include "dgt_packed.h"

namespace {

std::string json_escape(const std::string &s) {
    std::string o;
    for (char c : s) {
        if (c == '"' || c == '\\') { o += '\\'; o += c; }
        else if ((unsigned char)c < 0x20) { char b[8]; std::snprintf(b, sizeof b, "\\u%04x", c); o += b; }
        else o += c;
    }
    return o;
}

// ---- a small JSON reader for the header (objects, arrays, strings, integers)
struct JVal {
    enum Kind { NUL, NUM, STR, ARR, OBJ } kind = NUL;
    uint64_t num = 0;
    std::string str;
    std::vector<JVal> arr;
    std::map<std::string, JVal> obj;
};

struct JParser {
    const char *p, *e;
    int depth = 0;
    bool ok = true;
    void ws() { while (p < e && (*p == ' ' || *p == '\n' || *p == '\r' || *p == '\t')) p++; }
    bool str(std::string &out) {
        if (p >= e || *p != '"') return false;
        p++;
        while (p < e && *p != '"') {
            if (*p == '\\') {
                p++;
                if (p >= e) return false;
                if (*p == 'u') {
                    if (e - p < 5) return false;
                    unsigned v = (unsigned)std::strtoul(std::string(p + 1, p + 5).c_str(), nullptr, 16);
                    out += (char)(v & 0x7F);
                    p += 5;
                    continue;
                }
                out += *p == 'n' ? '\n' : *p == 't' ? '\t' : *p;
                p++;
            } else {
                out += *p++;
            }
        }
        if (p >= e) return false;
        p++;
        return true;
    }
    bool val(JVal &v) {
        if (++depth > 16) return false;
        ws();
        if (p >= e) return false;
        bool r = true;
        if (*p == '{') {
            v.kind = JVal::OBJ;
            p++;
            ws();
            if (p < e && *p == '}') { p++; depth--; return true; }
            for (;;) {
                ws();
                std::string k;
                if (!str(k)) { r = false; break; }
                ws();
                if (p >= e || *p != ':') { r = false; break; }
                p++;
                JVal c;
                if (!val(c)) { r = false; break; }
                v.obj[k] = std::move(c);
                ws();
                if (p < e && *p == ',') { p++; continue; }
                if (p < e && *p == '}') { p++; break; }
                r = false;
                break;
            }
        } else if (*p == '[') {
            v.kind = JVal::ARR;
            p++;
            ws();
            if (p < e && *p == ']') { p++; depth--; return true; }
            for (;;) {
                JVal c;
                if (!val(c)) { r = false; break; }
                v.arr.push_back(std::move(c));
                ws();
                if (p < e && *p == ',') { p++; continue; }
                if (p < e && *p == ']') { p++; break; }
                r = false;
                break;
            }
        } else if (*p == '"') {
            v.kind = JVal::STR;
            r = str(v.str);
        } else if (*p >= '0' && *p <= '9') {
            v.kind = JVal::NUM;
            uint64_t x = 0;
            while (p < e && *p >= '0' && *p <= '9') {
                if (x > (UINT64_MAX - 9) / 10) return false;
                x = x * 10 + (uint64_t)(*p++ - '0');
            }
            v.num = x;
        } else {
            r = false;
        }
        depth--;
        return r;
    }
};

struct Arr {
    std::string name;
    const void *data;
    uint64_t bytes;
};

void arrays_of(const dgt_packed *t, const std::string &x, std::vector<Arr> &out) {
    const dgt_packed_view &v = t->v;
    out.push_back({x + ".sm", t->sm.data(), t->sm.size()});
    if (v.format == 2) {
        out.push_back({x + ".rice", t->words.data(), t->words.size() * 4});
        out.push_back({x + ".blkq", t->blkq.data(), t->blkq.size()});
        out.push_back({x + ".grp", t->grp.data(), t->grp.size() * 4});
    } else {
        out.push_back({x + ".f1", t->payload.data(), t->payload.size()});
        out.push_back({x + ".tw", t->tw.data(), t->tw.size()});
        out.push_back({x + ".tesc", t->tesc.data(), t->tesc.size()});
        out.push_back({x + ".esc1", t->esc1.data(), t->esc1.size()});
        out.push_back({x + ".grp1", t->grp1.data(), t->grp1.size() * 4});
    }
}

std::string meta_of(const dgt_packed *t) {
    const dgt_packed_view &v = t->v;
    char buf[256];
    std::snprintf(buf, sizeof buf, "format=%d;rows=%llu;cols=%llu;k=%d;T=%d;n_esc15=%llu;table=",
                  v.format, (unsigned long long)v.rows, (unsigned long long)v.cols, v.rice_k,
                  v.n_table, (unsigned long long)v.n_esc15);
    std::string s = buf;
    for (int i = 0; i < v.n_table; i++) {
        std::snprintf(buf, sizeof buf, "%02x", v.table[i]);
        s += buf;
    }
    return s;
}

bool parse_meta(const std::string &s, dgt_packed_view &v) {
    std::map<std::string, std::string> kv;
    size_t i = 0;
    while (i < s.size()) {
        size_t j = s.find(';', i);
        if (j == std::string::npos) j = s.size();
        std::string item = s.substr(i, j - i);
        size_t q = item.find('=');
        if (q == std::string::npos) return false;
        kv[item.substr(0, q)] = item.substr(q + 1);
        i = j + 1;
    }
    const char *keys[] = {"format", "rows", "cols", "k", "T", "n_esc15", "table"};
    for (const char *k : keys)
        if (!kv.count(k)) return false;
    char *end = nullptr;
    v.format = (int)std::strtol(kv["format"].c_str(), &end, 10);
    v.rows = std::strtoull(kv["rows"].c_str(), &end, 10);
    v.cols = std::strtoull(kv["cols"].c_str(), &end, 10);
    v.rice_k = (int)std::strtol(kv["k"].c_str(), &end, 10);
    v.n_table = (int)std::strtol(kv["T"].c_str(), &end, 10);
    v.n_esc15 = std::strtoull(kv["n_esc15"].c_str(), &end, 10);
    const std::string &tab = kv["table"];
    if ((v.format != 1 && v.format != 2) || v.n_table < 0 || v.n_table > 256 ||
        tab.size() != 2 * (size_t)v.n_table || v.rice_k < 0 || v.rice_k > 7)
        return false;
    if (v.rows && (v.rows * v.cols) / v.rows != v.cols) return false;
    std::memset(v.table, 0, 256);
    for (int t = 0; t < v.n_table; t++)
        v.table[t] = (uint8_t)std::strtoul(tab.substr(2 * t, 2).c_str(), nullptr, 16);
    return true;
}

}  // namespace

extern "C" {

int dgt_write(const char *path, const dgt_packed *const *tensors, const char *const *names,
              int count) {
    if (!path || count < 0 || (count && (!tensors || !names))) return DGT_ERR_ARG;
    std::vector<Arr> arrs;
    std::string meta = "\"__metadata__\":{";
    for (int i = 0; i < count; i++) {
        if (!tensors[i] || !names[i] || !names[i][0]) return DGT_ERR_ARG;
        arrays_of(tensors[i], names[i], arrs);
        if (i) meta += ",";
        meta += "\"" + json_escape(names[i]) + "\":\"" + json_escape(meta_of(tensors[i])) + "\"";
    }
    meta += "}";
    std::string hdr = "{" + meta;
    uint64_t off = 0;
    char buf[128];
    for (const Arr &a : arrs) {
        std::snprintf(buf, sizeof buf, "\"dtype\":\"U8\",\"shape\":[%llu],\"data_offsets\":[%llu,%llu]}",
                      (unsigned long long)a.bytes, (unsigned long long)off,
                      (unsigned long long)(off + a.bytes));
        hdr += ",\"" + json_escape(a.name) + "\":{" + buf;
        off += a.bytes;
    }
    hdr += "}";
    while (hdr.size() % 8) hdr += ' ';
    // Written to a temporary file beside the target and renamed over it once
    // complete, so a failed or interrupted write never leaves a partial
    // container under `path`.
    const std::string tmp = std::string(path) + ".tmp" + std::to_string((long long)getpid());
    FILE *f = std::fopen(tmp.c_str(), "wb");
    if (!f) return DGT_ERR_IO;
    uint64_t hl = hdr.size();
    uint8_t le[8];
    for (int i = 0; i < 8; i++) le[i] = (uint8_t)(hl >> (8 * i));
    bool ok = std::fwrite(le, 1, 8, f) == 8 && std::fwrite(hdr.data(), 1, hdr.size(), f) == hdr.size();
    for (const Arr &a : arrs)
        if (ok && a.bytes) ok = std::fwrite(a.data, 1, a.bytes, f) == a.bytes;
    ok = (std::fclose(f) == 0) && ok;
    ok = ok && std::rename(tmp.c_str(), path) == 0;
    if (!ok) std::remove(tmp.c_str());
    return ok ? DGT_OK : DGT_ERR_IO;
}

int dgt_read(const char *path, dgt_packed ***tensors, char ***names, int *count) {
    if (!path || !tensors || !names || !count) return DGT_ERR_ARG;
    *tensors = nullptr;
    *names = nullptr;
    *count = 0;
    FILE *f = std::fopen(path, "rb");
    if (!f) return DGT_ERR_IO;
    std::unique_ptr<FILE, int (*)(FILE *)> guard(f, std::fclose);
    uint8_t le[8];
    if (std::fread(le, 1, 8, f) != 8) return DGT_ERR_CORRUPT;
    uint64_t hl = 0;
    for (int i = 0; i < 8; i++) hl |= (uint64_t)le[i] << (8 * i);
    if (hl > (64u << 20)) return DGT_ERR_CORRUPT;
    if (fseeko(f, 0, SEEK_END) != 0) return DGT_ERR_IO;
    const off_t fsz = ftello(f);
    if (fsz < 0 || (uint64_t)fsz < 8 + hl) return DGT_ERR_CORRUPT;
    const uint64_t dsz = (uint64_t)fsz - 8 - hl;
    if (fseeko(f, 8, SEEK_SET) != 0) return DGT_ERR_IO;
    std::string hdr(hl, '\0');
    if (hl && std::fread(&hdr[0], 1, hl, f) != hl) return DGT_ERR_CORRUPT;
    JParser jp{hdr.data(), hdr.data() + hdr.size()};
    JVal root;
    if (!jp.val(root) || root.kind != JVal::OBJ) return DGT_ERR_CORRUPT;
    auto mit = root.obj.find("__metadata__");
    if (mit == root.obj.end() || mit->second.kind != JVal::OBJ) return DGT_ERR_CORRUPT;
    // Each array is read from the file straight into its destination (no
    // whole-file buffer): its byte range [a, b) of the data section.
    bool oom = false;
    auto span = [&](const std::string &nm, uint64_t *a, uint64_t *b) -> bool {
        auto it = root.obj.find(nm);
        if (it == root.obj.end() || it->second.kind != JVal::OBJ) return false;
        auto &o = it->second.obj;
        auto d = o.find("data_offsets");
        if (d == o.end() || d->second.kind != JVal::ARR || d->second.arr.size() != 2) return false;
        *a = d->second.arr[0].num;
        *b = d->second.arr[1].num;
        return *a <= *b && *b <= dsz;
    };
    auto fill = [&](uint64_t a, void *dst, uint64_t bytes) -> bool {
        if (bytes == 0) return true;
        if (fseeko(f, (off_t)(8 + hl + a), SEEK_SET) != 0) return false;
        return std::fread(dst, 1, bytes, f) == bytes;
    };
    auto get = [&](const std::string &nm, auto &dst) -> bool {
        uint64_t a, b;
        if (!span(nm, &a, &b)) return false;
        try {
            dst.resize(b - a);
        } catch (const std::bad_alloc &) {
            oom = true;
            return false;
        }
        return fill(a, dst.data(), b - a);
    };
    auto get32 = [&](const std::string &nm, std::vector<uint32_t> &dst) -> bool {
        uint64_t a, b;
        if (!span(nm, &a, &b) || (b - a) % 4) return false;
        try {
            dst.resize((b - a) / 4);
        } catch (const std::bad_alloc &) {
            oom = true;
            return false;
        }
        return fill(a, dst.data(), b - a);
    };
    std::vector<dgt_packed *> out;
    std::vector<std::string> nms;
    int rc = DGT_OK;
    for (auto &kv : mit->second.obj) {
        if (kv.second.kind != JVal::STR) { rc = DGT_ERR_CORRUPT; break; }
        dgt_packed *t = new (std::nothrow) dgt_packed();
        if (!t) { rc = DGT_ERR_OOM; break; }
        std::memset(&t->v, 0, sizeof(t->v));
        const std::string &x = kv.first;
        bool ok = parse_meta(kv.second.str, t->v) && get(x + ".sm", t->sm);
        const uint64_t n = t->v.rows * t->v.cols;
        ok = ok && t->sm.size() == n;
        if (ok && t->v.format == 2) {
            uint64_t nblk = (n + DGT_BLOCK - 1) / DGT_BLOCK, ngrp = (nblk + DGT_GROUP - 1) / DGT_GROUP;
            ok = get32(x + ".rice", t->words) && get(x + ".blkq", t->blkq) &&
                 get32(x + ".grp", t->grp) && t->blkq.size() == nblk && t->grp.size() == 2 * ngrp;
            for (uint64_t g = 0; ok && g < ngrp; g++) ok = t->grp[2 * g] <= t->words.size();
        } else if (ok) {
            uint64_t nt = (n + DGT_TILE - 1) / DGT_TILE, ngrp = (nt + DGT_GROUP - 1) / DGT_GROUP;
            ok = get(x + ".f1", t->payload) && get(x + ".tw", t->tw) && get(x + ".tesc", t->tesc) &&
                 get(x + ".esc1", t->esc1) && get32(x + ".grp1", t->grp1) && t->tw.size() == nt &&
                 t->tesc.size() == nt && t->grp1.size() == 3 * ngrp;
        }
        if (!ok) {
            delete t;
            rc = oom ? DGT_ERR_OOM : DGT_ERR_CORRUPT;
            break;
        }
        t->refresh();
        out.push_back(t);
        nms.push_back(x);
    }
    if (rc != DGT_OK) {
        for (auto *t : out) delete t;
        return rc;
    }
    int c = (int)out.size();
    dgt_packed **ta = (dgt_packed **)std::calloc(c ? c : 1, sizeof(dgt_packed *));
    char **na = (char **)std::calloc(c ? c : 1, sizeof(char *));
    if (!ta || !na) {
        std::free(ta);
        std::free(na);
        for (auto *t : out) delete t;
        return DGT_ERR_OOM;
    }
    for (int i = 0; i < c; i++) {
        na[i] = (char *)std::malloc(nms[i].size() + 1);
        if (!na[i]) {
            for (int j = 0; j < i; j++) std::free(na[j]);
            std::free(ta);
            std::free(na);
            for (auto *t : out) delete t;
            return DGT_ERR_OOM;
        }
        std::memcpy(na[i], nms[i].c_str(), nms[i].size() + 1);
        ta[i] = out[i];
    }
    *tensors = ta;
    *names = na;
    *count = c;
    return DGT_OK;
}

void dgt_read_free(dgt_packed **tensors, char **names, int count) {
    for (int i = 0; i < count; i++) {
        if (tensors) delete tensors[i];
        if (names) std::free(names[i]);
    }
    std::free(tensors);
    std::free(names);
}

}  // extern "C"
