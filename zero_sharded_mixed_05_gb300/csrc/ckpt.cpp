// ckpt.cpp -- sharded checkpoint files and their consolidation (host only).
//
// One file per rank holds that rank's real fp32 master weights, m and v and
// its loss-scaler state; zero_opt_consolidate_fp32 merges the files of all
// ranks into the full fp32 weights with the padding dropped.  The format is
// documented beside the declarations in include/zero_opt.h.
#include <cerrno>
#include <cstdio>
#include <cstring>
#include <memory>
#include <vector>

#include "host_util.h"
#include "zero_opt.h"

namespace {

const char kMagic[8] = {'Z', 'O', 'P', 'T', 'S', 'H', 'D', '1'};
constexpr uint32_t kVersion = 1;
// magic, version, reserved, numel, world, rank, begin, real_len, scale,
// last_skipped, clean_steps, t, skipped_total, overflows, reserved, checksum
constexpr long kHeaderBytes = 8 + 4 + 4 + 8 + 4 + 4 + 8 + 8 + 4 + 4 + 8 + 8 + 8 + 4 + 4 + 8;

// 64-bit FNV-1a over 8-byte little-endian words of a byte stream fed in
// pieces; a trailing partial word is zero-extended.
struct WordHash {
  uint64_t h = 0xcbf29ce484222325ull;
  unsigned char pend[8];
  size_t npend = 0;
  void word(uint64_t w) {
    h ^= w;
    h *= 0x100000001b3ull;
  }
  void feed(const void* data, size_t n) {
    const unsigned char* p = static_cast<const unsigned char*>(data);
    while (n > 0 && npend > 0) {
      pend[npend++] = *p++;
      --n;
      if (npend == 8) {
        uint64_t w;
        std::memcpy(&w, pend, 8);
        word(w);
        npend = 0;
      }
    }
    for (; n >= 8; n -= 8, p += 8) {
      uint64_t w;
      std::memcpy(&w, p, 8);
      word(w);
    }
    while (n > 0) {
      pend[npend++] = *p++;
      --n;
    }
  }
  uint64_t finish() {
    if (npend > 0) {
      uint64_t w = 0;
      std::memcpy(&w, pend, npend);
      word(w);
      npend = 0;
    }
    return h;
  }
};

struct FileCloser {
  void operator()(FILE* f) const {
    if (f) std::fclose(f);
  }
};
using File = std::unique_ptr<FILE, FileCloser>;

template <typename T>
bool put(FILE* f, T v) {
  return std::fwrite(&v, sizeof(T), 1, f) == 1;
}
template <typename T>
bool get(FILE* f, T* v) {
  return std::fread(v, sizeof(T), 1, f) == 1;
}

zero_status check_info(const zero_opt_ckpt_info* in) {
  if (in->numel < 0 || in->world < 1 || in->rank < 0 || in->rank >= in->world)
    return zo::fail(ZERO_EINVAL, "checkpoint info: bad numel/world/rank");
  int64_t begin, real, shard;
  zo::shard_range(in->numel, in->world, in->rank, &begin, &real, &shard);
  if (in->begin != begin || in->real_len != real)
    return zo::fail(ZERO_EINVAL, "checkpoint info: begin/real_len are not rank %d's shard",
                    in->rank);
  return ZERO_OK;
}

bool write_floats(FILE* f, const float* a, int64_t n) {
  const int64_t kChunk = 1 << 20;
  for (int64_t i = 0; i < n; i += kChunk) {
    const int64_t c = n - i < kChunk ? n - i : kChunk;
    if (std::fwrite(a + i, sizeof(float), (size_t)c, f) != (size_t)c) return false;
  }
  return true;
}

bool read_floats(FILE* f, float* a, int64_t n, WordHash* hs) {
  const int64_t kChunk = 1 << 20;
  for (int64_t i = 0; i < n; i += kChunk) {
    const int64_t c = n - i < kChunk ? n - i : kChunk;
    if (std::fread(a + i, sizeof(float), (size_t)c, f) != (size_t)c) return false;
    hs->feed(a + i, sizeof(float) * (size_t)c);
  }
  return true;
}

}  // namespace

extern "C" {

zero_status zero_opt_ckpt_write(const char* path, const zero_opt_ckpt_info* info,
                                const float* master, const float* m, const float* v) {
  if (!path || !info) return zo::fail(ZERO_EINVAL, "path and info must be non-NULL");
  zero_status st = check_info(info);
  if (st != ZERO_OK) return st;
  if (info->real_len > 0 && (!master || !m || !v))
    return zo::fail(ZERO_EINVAL, "master, m and v must be non-NULL");
  const size_t bytes = sizeof(float) * (size_t)info->real_len;
  WordHash hs;
  if (bytes > 0) {
    hs.feed(master, bytes);
    hs.feed(m, bytes);
    hs.feed(v, bytes);
  }
  const uint64_t sum = hs.finish();
  File f(std::fopen(path, "wb"));
  if (!f) return zo::fail(ZERO_EINVAL, "cannot open %s: %s", path, std::strerror(errno));
  const zero_opt_scaler_state& s = info->scaler;
  bool ok = std::fwrite(kMagic, 1, 8, f.get()) == 8 && put<uint32_t>(f.get(), kVersion) &&
            put<uint32_t>(f.get(), 0) && put(f.get(), info->numel) &&
            put(f.get(), info->world) && put(f.get(), info->rank) &&
            put(f.get(), info->begin) && put(f.get(), info->real_len) &&
            put(f.get(), s.scale) && put(f.get(), s.last_skipped) &&
            put(f.get(), s.clean_steps) && put(f.get(), s.t) &&
            put(f.get(), s.skipped_total) && put(f.get(), s.overflows) &&
            put<int32_t>(f.get(), 0) && put(f.get(), sum);
  ok = ok && write_floats(f.get(), master, info->real_len) &&
       write_floats(f.get(), m, info->real_len) && write_floats(f.get(), v, info->real_len);
  if (!ok) return zo::fail(ZERO_EINVAL, "write to %s failed: %s", path, std::strerror(errno));
  if (std::fclose(f.release()) != 0)
    return zo::fail(ZERO_EINVAL, "closing %s failed: %s", path, std::strerror(errno));
  return ZERO_OK;
}

zero_status zero_opt_ckpt_read(const char* path, zero_opt_ckpt_info* info, float* master,
                               float* m, float* v) {
  if (!path || !info) return zo::fail(ZERO_EINVAL, "path and info must be non-NULL");
  File f(std::fopen(path, "rb"));
  if (!f) return zo::fail(ZERO_EINVAL, "cannot open %s: %s", path, std::strerror(errno));
  char magic[8];
  uint32_t version = 0, reserved = 0;
  int32_t reserved2 = 0;
  uint64_t sum = 0;
  zero_opt_ckpt_info in;
  std::memset(&in, 0, sizeof(in));
  zero_opt_scaler_state& s = in.scaler;
  const bool ok = std::fread(magic, 1, 8, f.get()) == 8 && get(f.get(), &version) &&
                  get(f.get(), &reserved) && get(f.get(), &in.numel) &&
                  get(f.get(), &in.world) && get(f.get(), &in.rank) &&
                  get(f.get(), &in.begin) && get(f.get(), &in.real_len) &&
                  get(f.get(), &s.scale) && get(f.get(), &s.last_skipped) &&
                  get(f.get(), &s.clean_steps) && get(f.get(), &s.t) &&
                  get(f.get(), &s.skipped_total) && get(f.get(), &s.overflows) &&
                  get(f.get(), &reserved2) && get(f.get(), &sum);
  if (!ok) return zo::fail(ZERO_EINVAL, "%s: truncated header", path);
  if (std::memcmp(magic, kMagic, 8) != 0) return zo::fail(ZERO_EINVAL, "%s: not a shard file", path);
  if (version != kVersion) return zo::fail(ZERO_EINVAL, "%s: unknown version %u", path, version);
  zero_status st = check_info(&in);
  if (st != ZERO_OK) return st;
  if (std::fseek(f.get(), 0, SEEK_END) != 0) return zo::fail(ZERO_EINVAL, "%s: cannot seek", path);
  const long size = std::ftell(f.get());
  if (size != kHeaderBytes + 12 * (long)in.real_len)
    return zo::fail(ZERO_EINVAL, "%s: size %ld does not match its header", path, size);
  *info = in;
  if (!master && !m && !v) return ZERO_OK;
  std::fseek(f.get(), kHeaderBytes, SEEK_SET);
  std::vector<float> scratch;
  WordHash hs;
  float* dst[3] = {master, m, v};
  for (int k = 0; k < 3; ++k) {
    float* d = dst[k];
    if (!d) {
      scratch.resize((size_t)in.real_len);
      d = scratch.data();
    }
    if (!read_floats(f.get(), d, in.real_len, &hs))
      return zo::fail(ZERO_EINVAL, "%s: truncated payload", path);
  }
  if (hs.finish() != sum) return zo::fail(ZERO_EINVAL, "%s: checksum mismatch", path);
  return ZERO_OK;
}

zero_status zero_opt_consolidate_fp32(const char* const* paths, int32_t n_paths,
                                      int64_t numel, float* out) {
  if (!paths || n_paths < 1 || numel < 0 || (numel > 0 && !out))
    return zo::fail(ZERO_EINVAL, "bad arguments");
  std::vector<char> seen((size_t)n_paths, 0);
  std::vector<float> tmp_m, tmp_v;
  for (int32_t i = 0; i < n_paths; ++i) {
    if (!paths[i]) return zo::fail(ZERO_EINVAL, "path %d is NULL", i);
    zero_opt_ckpt_info in;
    zero_status st = zero_opt_ckpt_read(paths[i], &in, nullptr, nullptr, nullptr);
    if (st != ZERO_OK) return st;
    if (in.numel != numel || in.world != n_paths)
      return zo::fail(ZERO_EINVAL, "%s: numel %lld / world %d do not match %lld / %d", paths[i],
                      (long long)in.numel, in.world, (long long)numel, n_paths);
    if (seen[in.rank]) return zo::fail(ZERO_EINVAL, "rank %d appears twice", in.rank);
    seen[in.rank] = 1;
    tmp_m.resize((size_t)in.real_len + 1);
    tmp_v.resize((size_t)in.real_len + 1);
    float* dst = in.real_len > 0 ? out + in.begin : tmp_m.data();
    st = zero_opt_ckpt_read(paths[i], &in, dst, tmp_m.data(), tmp_v.data());
    if (st != ZERO_OK) return st;
  }
  return ZERO_OK;
}

}  // extern "C"
