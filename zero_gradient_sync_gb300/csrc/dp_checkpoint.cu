// Sharded checkpoints of the optimizer state, with resharding on load.
//
// "Distributed Training: Split along the Four Axes" -- checkpoint paragraphs: under ZeRO/FSDP the state is
// stored in shards by rank; a checkpoint either reshards to a different world size or says it cannot; it is
// written as temporary artifacts plus an atomic manifest, so a save that half fails leaves no corrupted
// snapshot; loss scaling and parallel metadata belong in it.
//
// Layout on disk, under root/:
//   <tag>/shard_<r>.bin   rank r's master, m, v (its dp_shard_len elements each, fp32, in local order)
//   <tag>/state.bin       the step state (t, beta powers, loss scale, good_steps; work fields zeroed)
//   <tag>/layout.bin      the layout the shards were written with (stage, n, psi, segments)
//   <tag>/user.bin        the caller's opaque metadata (LR schedule, RNG, data cursor, ...), possibly empty
//   <tag>/MANIFEST        one line per file: name, bytes, FNV-1a 64 checksum
//   LATEST                the tag of the newest complete checkpoint
// A save writes <tag>.partial/, syncs every file, renames it to <tag>/, then replaces LATEST by rename.
// Shard files are written and read by a few host threads at once, each with its own pinned chunk and CUDA
// stream, since one thread's buffered file writes run far below the host-device link.
#include <ctype.h>
#include <errno.h>
#include <fcntl.h>
#include <stdio.h>
#include <string.h>
#include <sys/stat.h>
#include <sys/types.h>
#include <unistd.h>

#include <algorithm>
#include <atomic>
#include <string>
#include <thread>
#include <vector>

#include "dp_internal.h"
#include "dpstep.h"

namespace {

constexpr uint32_t SHARD_MAGIC = 0x48535044u;   // "DPSH"
constexpr uint32_t LAYOUT_MAGIC = 0x4C535044u;  // "DPSL"
constexpr size_t CHUNK = size_t(1) << 24;       // bytes per host staging chunk

// Checksum: FNV-1a 64 (Fowler, Noll, Vo; offset basis 14695981039346656037, prime 1099511628211) taken over
// the file as little-endian 64-bit words, the last 0..7 bytes one at a time.  Word steps keep a checksum pass
// near memory speed; byte steps would cost a multiply per byte.
constexpr uint64_t FNV_BASIS = 14695981039346656037ull, FNV_PRIME = 1099511628211ull;

struct Fnv64 {
  uint64_t h = FNV_BASIS;
  unsigned char pend[8];
  int np = 0;
  static uint64_t le64(const unsigned char* b) {
    uint64_t w = 0;
    for (int i = 7; i >= 0; --i) w = (w << 8) | b[i];
    return w;
  }
  void word(uint64_t w) {
    h ^= w;
    h *= FNV_PRIME;
  }
  void add(const void* p, size_t n) {
    const unsigned char* b = static_cast<const unsigned char*>(p);
    while (np && n) {
      pend[np++] = *b++;
      --n;
      if (np == 8) {
        word(le64(pend));
        np = 0;
      }
    }
    for (; n >= 8; b += 8, n -= 8) word(le64(b));
    while (n) {
      pend[np++] = *b++;
      --n;
    }
  }
  uint64_t digest() const {
    uint64_t x = h;
    for (int i = 0; i < np; ++i) {
      x ^= pend[i];
      x *= FNV_PRIME;
    }
    return x;
  }
};

struct Err {
  dp_status_t code = DP_OK;
  std::string msg;
  bool set(dp_status_t c, const std::string& m) {
    if (code == DP_OK) {
      code = c;
      msg = m;
    }
    return false;
  }
};

bool write_all(int fd, const void* p, size_t n, Fnv64* h, Err& err, const std::string& what) {
  const char* b = static_cast<const char*>(p);
  while (n) {
    ssize_t w = ::write(fd, b, n);
    if (w < 0) {
      if (errno == EINTR) continue;
      return err.set(DP_ERR_IO, "write " + what + ": " + strerror(errno));
    }
    if (h) h->add(b, (size_t)w);
    b += w;
    n -= (size_t)w;
  }
  return true;
}

bool read_at(int fd, void* p, size_t n, uint64_t off, Err& err, const std::string& what) {
  char* b = static_cast<char*>(p);
  while (n) {
    ssize_t r = ::pread(fd, b, n, (off_t)off);
    if (r < 0) {
      if (errno == EINTR) continue;
      return err.set(DP_ERR_IO, "read " + what + ": " + strerror(errno));
    }
    if (r == 0) return err.set(DP_ERR_IO, "read " + what + ": file too short");
    b += r;
    n -= (size_t)r;
    off += (uint64_t)r;
  }
  return true;
}

bool fsync_path(const std::string& path, Err& err) {
  int fd = ::open(path.c_str(), O_RDONLY);
  if (fd < 0) return err.set(DP_ERR_IO, "open " + path + ": " + strerror(errno));
  int rc = ::fsync(fd);
  ::close(fd);
  if (rc != 0) return err.set(DP_ERR_IO, "fsync " + path + ": " + strerror(errno));
  return true;
}

// Moves data between the caller's buffers (device memory, or host memory when host_buffers is set) and a
// host chunk.  Device copies go through this worker's pinned chunk on this worker's own stream; the caller's
// stream has been synchronised before any worker starts.
struct Stager {
  int host_buffers;
  cudaStream_t stream = nullptr;
  bool own_stream = true;
  float* pinned = nullptr;
  std::vector<float> pageable;
  explicit Stager(int hb) : host_buffers(hb) {}
  Stager(int hb, cudaStream_t s) : host_buffers(hb), stream(s), own_stream(false) {}
  Stager(const Stager&) = delete;
  ~Stager() {
    if (pinned) cudaFreeHost(pinned);
    if (stream && own_stream) cudaStreamDestroy(stream);
  }
  float* chunk(Err& err) {
    if (host_buffers) {
      pageable.resize(CHUNK / sizeof(float));
      return pageable.data();
    }
    if (!stream && own_stream) {
      cudaError_t e = cudaStreamCreateWithFlags(&stream, cudaStreamNonBlocking);
      if (e != cudaSuccess) {
        stream = nullptr;
        err.set(DP_ERR_CUDA, std::string("cudaStreamCreateWithFlags: ") + cudaGetErrorString(e));
        return nullptr;
      }
    }
    if (!pinned) {
      cudaError_t e = cudaMallocHost((void**)&pinned, CHUNK);
      if (e != cudaSuccess) {
        pinned = nullptr;
        err.set(DP_ERR_CUDA, std::string("cudaMallocHost: ") + cudaGetErrorString(e));
      }
    }
    return pinned;
  }
  bool out(void* host, const void* src, size_t bytes, Err& err) {
    if (host_buffers) {
      memcpy(host, src, bytes);
      return true;
    }
    cudaError_t e = cudaMemcpyAsync(host, src, bytes, cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return err.set(DP_ERR_CUDA, std::string("copy to host: ") + cudaGetErrorString(e));
    return true;
  }
  bool in(void* dst, const void* host, size_t bytes, Err& err) {
    if (host_buffers) {
      memcpy(dst, host, bytes);
      return true;
    }
    cudaError_t e = cudaMemcpyAsync(dst, host, bytes, cudaMemcpyHostToDevice, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return err.set(DP_ERR_CUDA, std::string("copy to device: ") + cudaGetErrorString(e));
    return true;
  }
};

// Runs fn(item, worker_index) for item = 0..count-1 on up to max_workers threads; returns the first error.
template <class F>
Err parallel_items(int64_t count, int max_workers, F fn) {
  const int w = (int)std::max<int64_t>(1, std::min<int64_t>(count, max_workers));
  std::vector<Err> errs(w);
  std::atomic<int64_t> next{0};
  std::atomic<int> failed{0};
  auto body = [&](int k) {
    for (;;) {
      if (failed.load()) return;
      const int64_t i = next.fetch_add(1);
      if (i >= count) return;
      if (!fn(i, k, errs[k])) {
        failed.store(1);
        return;
      }
    }
  };
  std::vector<std::thread> th;
  for (int k = 1; k < w; ++k) th.emplace_back(body, k);
  body(0);
  for (auto& t : th) t.join();
  for (Err& e : errs)
    if (e.code != DP_OK) return e;
  return Err{};
}

int io_workers() {
  const unsigned hc = std::thread::hardware_concurrency();
  return (int)std::max(1u, std::min(hc ? hc : 1u, 8u));
}

struct Seg {
  int64_t goff, len;
  int32_t owner;
  int64_t loff;
};

bool layout_segments(const dp_layout_t* L, std::vector<Seg>& segs, std::vector<int64_t>& shard_len, Err& err) {
  if (dp_layout_validate(L) != DP_OK) return err.set(DP_ERR_INVALID_ARG, dp_last_error());
  segs.clear();
  shard_len.assign(L->n, 0);
  for (int i = 0; i < L->nseg; ++i) {
    const dp_segment_t& s = L->seg[i];
    if (s.len == 0) continue;
    segs.push_back({s.global_off, s.len, s.owner, s.local_off});
    shard_len[s.owner] = std::max(shard_len[s.owner], s.local_off + s.len);
  }
  return true;
}

// Writes one file under dir, returning its size and checksum for the manifest.
struct FileOut {
  std::string path;
  int fd = -1;
  Fnv64 h;
  uint64_t bytes = 0;
  bool open(const std::string& p, Err& err) {
    path = p;
    fd = ::open(p.c_str(), O_WRONLY | O_CREAT | O_TRUNC, 0644);
    if (fd < 0) return err.set(DP_ERR_IO, "create " + p + ": " + strerror(errno));
    return true;
  }
  bool put(const void* b, size_t n, Err& err) {
    bytes += n;
    return write_all(fd, b, n, &h, err, path);
  }
  bool close(Err& err) {
    bool ok = true;
    if (::fsync(fd) != 0) ok = err.set(DP_ERR_IO, "fsync " + path + ": " + strerror(errno));
    ::close(fd);
    fd = -1;
    return ok;
  }
};

std::string base_name(const std::string& p) {
  size_t k = p.find_last_of('/');
  return k == std::string::npos ? p : p.substr(k + 1);
}

bool valid_tag(const char* tag) {
  if (!tag || !*tag || strlen(tag) > 200) return false;
  for (const char* c = tag; *c; ++c)
    if (!(isalnum((unsigned char)*c) || *c == '_' || *c == '-' || *c == '.')) return false;
  return tag[0] != '.';
}

struct ManifestEntry {
  std::string name;
  uint64_t bytes;
  uint64_t fnv;
};

bool read_manifest(const std::string& dir, std::vector<ManifestEntry>& out, Err& err) {
  FILE* f = fopen((dir + "/MANIFEST").c_str(), "r");
  if (!f) return err.set(DP_ERR_IO, "no MANIFEST in " + dir);
  char line[512];
  out.clear();
  bool header = false;
  while (fgets(line, sizeof(line), f)) {
    if (!header) {
      header = strncmp(line, "dpstep-checkpoint 1", 19) == 0;
      if (!header) break;
      continue;
    }
    char name[256];
    unsigned long long bytes = 0, fnv = 0;
    if (sscanf(line, "file %255s %llu %llx", name, &bytes, &fnv) == 3) out.push_back({name, bytes, fnv});
  }
  fclose(f);
  if (!header) return err.set(DP_ERR_IO, "MANIFEST of " + dir + " is not a checkpoint manifest");
  return true;
}

bool verify_file(const std::string& path, const ManifestEntry& e, Err& err) {
  int fd = ::open(path.c_str(), O_RDONLY);
  if (fd < 0) return err.set(DP_ERR_IO, "open " + path + ": " + strerror(errno));
  std::vector<char> buf(CHUNK);
  Fnv64 h;
  uint64_t total = 0;
  for (;;) {
    ssize_t r = ::read(fd, buf.data(), buf.size());
    if (r < 0) {
      if (errno == EINTR) continue;
      ::close(fd);
      return err.set(DP_ERR_IO, "read " + path + ": " + strerror(errno));
    }
    if (r == 0) break;
    h.add(buf.data(), (size_t)r);
    total += (uint64_t)r;
  }
  ::close(fd);
  if (total != e.bytes || h.digest() != e.fnv) return err.set(DP_ERR_IO, "checksum or size mismatch in " + path);
  return true;
}

// The files a complete checkpoint of n shards must list in its manifest.
std::vector<std::string> required_files(int n) {
  std::vector<std::string> v;
  for (int r = 0; r < n; ++r) v.push_back("shard_" + std::to_string(r) + ".bin");
  v.push_back("state.bin");
  v.push_back("layout.bin");
  v.push_back("user.bin");
  return v;
}

constexpr int64_t SHARD_HDR = 16 + 8;  // magic, version, rank, 0, then the shard length

dp_status_t save(const char* root, const char* tag, const dp_layout_t* layout, float* const* master,
                 float* const* m, float* const* v, const dp_step_state_t* d_state, const void* user_meta,
                 uint64_t user_meta_bytes, int32_t host_buffers, cudaStream_t stream) {
  Err err;
  std::vector<Seg> segs;
  std::vector<int64_t> shard_len;
  if (!root || !*root || !valid_tag(tag)) return dp::report_error(DP_ERR_INVALID_ARG, "checkpoint: bad root or tag");
  if (!master || !m || !v || !d_state || (user_meta_bytes && !user_meta))
    return dp::report_error(DP_ERR_INVALID_ARG, "checkpoint: NULL argument");
  if (!layout_segments(layout, segs, shard_len, err)) return dp::report_error(err.code, err.msg.c_str());
  const int n = layout->n;
  const bool full = layout->stage == DP_STAGE_DP;
  for (int r = 0; r < n; ++r) {
    const int64_t need = full ? layout->psi : shard_len[r];
    if (need && (!master[r] || !m[r] || !v[r]))
      return dp::report_error(DP_ERR_INVALID_ARG, "checkpoint: NULL state array of a non-empty shard");
  }
  if (!host_buffers) {
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return dp::report_error(DP_ERR_CUDA, cudaGetErrorString(e));
  }
  const int64_t cap = (int64_t)(CHUNK / sizeof(float));

  const std::string final_dir = std::string(root) + "/" + tag;
  const std::string dir = final_dir + ".partial";
  struct stat st;
  if (::stat(final_dir.c_str(), &st) == 0)
    return dp::report_error(DP_ERR_IO, ("checkpoint: already exists: " + final_dir).c_str());
  if (::mkdir(root, 0755) != 0 && errno != EEXIST)
    return dp::report_error(DP_ERR_IO, (std::string("mkdir ") + root + ": " + strerror(errno)).c_str());
  if (::mkdir(dir.c_str(), 0755) != 0 && errno != EEXIST)
    return dp::report_error(DP_ERR_IO, ("mkdir " + dir + ": " + strerror(errno)).c_str());

  float* const* arrays[3] = {master, m, v};
  const int workers = io_workers();
  std::vector<Stager*> io;
  for (int k = 0; k < workers; ++k) io.push_back(new Stager(host_buffers));
  std::vector<FileOut> files(n);
  // shard_<r>.bin: header, then master, m, v of rank r's shard in local order (holes as zeros); one file per item
  err = parallel_items(n, workers, [&](int64_t r, int w, Err& e) {
    float* buf = io[w]->chunk(e);
    if (!buf) return false;
    std::vector<Seg> mine;
    for (const Seg& sg : segs)
      if (sg.owner == r) mine.push_back(sg);
    std::sort(mine.begin(), mine.end(), [](const Seg& x, const Seg& y) { return x.loff < y.loff; });
    FileOut& f = files[r];
    if (!f.open(dir + "/shard_" + std::to_string(r) + ".bin", e)) return false;
    const uint32_t hdr[4] = {SHARD_MAGIC, 1u, (uint32_t)r, 0u};
    const int64_t len = shard_len[r];
    f.put(hdr, sizeof(hdr), e);
    f.put(&len, sizeof(len), e);
    for (int k = 0; k < 3 && e.code == DP_OK; ++k) {
      int64_t written = 0;
      for (const Seg& sg : mine) {
        while (written < sg.loff && e.code == DP_OK) {
          const int64_t c = std::min(sg.loff - written, cap);
          memset(buf, 0, (size_t)c * 4);
          f.put(buf, (size_t)c * 4, e);
          written += c;
        }
        for (int64_t i = 0; i < sg.len && e.code == DP_OK;) {
          const int64_t c = std::min(sg.len - i, cap);
          // stage 0 keeps full-length arrays: rank r's chunk is read at its global index
          const float* src = arrays[k][r] + (full ? sg.goff : sg.loff) + i;
          if (io[w]->out(buf, src, (size_t)c * 4, e)) f.put(buf, (size_t)c * 4, e);
          i += c;
        }
        written = sg.loff + sg.len;
      }
    }
    f.close(e);
    return e.code == DP_OK;
  });
  for (Stager* x : io) delete x;
  Stager small(host_buffers, stream);  // the 64-byte state goes over the caller's stream
  // state.bin: the step state with the kernel-internal and per-step fields cleared
  if (err.code == DP_OK) {
    dp_step_state_t hs;
    if (small.out(&hs, d_state, sizeof(hs), err)) {
      hs.found_inf = 0;
      hs.nonfinite = 0;
      hs.work_count = 0;
      hs.work_found = 0;
      hs.work_ticket = 0;
      hs.cur_set = 0;
      FileOut f;
      if (f.open(dir + "/state.bin", err)) {
        f.put(&hs, sizeof(hs), err);
        f.close(err);
        files.push_back(f);
      }
    }
  }
  // layout.bin: header, psi, nseg, the segments as given
  if (err.code == DP_OK) {
    FileOut f;
    if (f.open(dir + "/layout.bin", err)) {
      const uint32_t hdr[4] = {LAYOUT_MAGIC, 1u, (uint32_t)layout->stage, (uint32_t)layout->n};
      const int64_t psi = layout->psi, nseg = layout->nseg;
      f.put(hdr, sizeof(hdr), err);
      f.put(&psi, 8, err);
      f.put(&nseg, 8, err);
      if (layout->nseg) f.put(layout->seg, sizeof(dp_segment_t) * (size_t)layout->nseg, err);
      f.close(err);
      files.push_back(f);
    }
  }
  if (err.code == DP_OK) {
    FileOut f;
    if (f.open(dir + "/user.bin", err)) {
      if (user_meta_bytes) f.put(user_meta, (size_t)user_meta_bytes, err);
      f.close(err);
      files.push_back(f);
    }
  }
  if (err.code == DP_OK) {
    FileOut f;
    if (f.open(dir + "/MANIFEST", err)) {
      std::string text = "dpstep-checkpoint 1\n";
      char line[400];
      for (const FileOut& x : files) {
        snprintf(line, sizeof(line), "file %s %llu %016llx\n", base_name(x.path).c_str(),
                 (unsigned long long)x.bytes, (unsigned long long)x.h.digest());
        text += line;
      }
      f.put(text.data(), text.size(), err);
      f.close(err);
    }
  }
  // publication: the directory appears under its name complete, then LATEST moves to it
  if (err.code == DP_OK) fsync_path(dir, err);
  if (err.code == DP_OK && ::rename(dir.c_str(), final_dir.c_str()) != 0)
    err.set(DP_ERR_IO, "rename " + dir + ": " + strerror(errno));
  if (err.code == DP_OK) fsync_path(root, err);
  if (err.code == DP_OK) {
    const std::string tmp = std::string(root) + "/LATEST.partial";
    FileOut f;
    if (f.open(tmp, err)) {
      const std::string t = std::string(tag) + "\n";
      f.put(t.data(), t.size(), err);
      f.close(err);
    }
    if (err.code == DP_OK && ::rename(tmp.c_str(), (std::string(root) + "/LATEST").c_str()) != 0)
      err.set(DP_ERR_IO, std::string("rename LATEST: ") + strerror(errno));
    if (err.code == DP_OK) fsync_path(root, err);
  }
  if (err.code != DP_OK) return dp::report_error(err.code, err.msg.c_str());
  return DP_OK;
}

bool resolve_tag(const char* root, const char* tag, std::string& out, Err& err) {
  if (tag) {
    if (!valid_tag(tag)) return err.set(DP_ERR_INVALID_ARG, "checkpoint: bad tag");
    out = tag;
    return true;
  }
  FILE* f = fopen((std::string(root) + "/LATEST").c_str(), "r");
  if (!f) return err.set(DP_ERR_IO, std::string("checkpoint: no LATEST under ") + root);
  char line[256] = {0};
  if (!fgets(line, sizeof(line), f)) line[0] = 0;
  fclose(f);
  out = line;
  while (!out.empty() && (out.back() == '\n' || out.back() == '\r')) out.pop_back();
  if (!valid_tag(out.c_str())) return err.set(DP_ERR_IO, "checkpoint: LATEST names no valid tag");
  return true;
}

// Reads and checks the saved layout; segs receives its segments (old.seg points into it).
bool read_layout(const std::string& dir, dp_layout_t& old, std::vector<dp_segment_t>& segs, Err& err) {
  int fd = ::open((dir + "/layout.bin").c_str(), O_RDONLY);
  if (fd < 0) return err.set(DP_ERR_IO, "checkpoint: no layout.bin in " + dir);
  uint32_t hdr[4];
  int64_t psi = 0, nseg = 0;
  bool ok = read_at(fd, hdr, sizeof(hdr), 0, err, "layout.bin") && read_at(fd, &psi, 8, 16, err, "layout.bin") &&
            read_at(fd, &nseg, 8, 24, err, "layout.bin");
  if (ok && (hdr[0] != LAYOUT_MAGIC || hdr[1] != 1u || nseg < 0 || nseg > DP_MAX_SEG))
    ok = err.set(DP_ERR_IO, "checkpoint: layout.bin is not a layout");
  if (ok) {
    segs.resize((size_t)nseg);
    if (nseg) ok = read_at(fd, segs.data(), sizeof(dp_segment_t) * (size_t)nseg, 32, err, "layout.bin");
  }
  ::close(fd);
  if (!ok) return false;
  old = dp_layout_t{(int32_t)hdr[2], (int32_t)hdr[3], psi, (int32_t)nseg, 0, segs.data()};
  return true;
}

bool open_checkpoint(const char* root, const char* tag, int verify, std::string& dir, dp_layout_t& old,
                     std::vector<dp_segment_t>& old_segs, uint64_t* user_bytes, Err& err) {
  std::string t;
  if (!resolve_tag(root, tag, t, err)) return false;
  dir = std::string(root) + "/" + t;
  std::vector<ManifestEntry> man;
  if (!read_manifest(dir, man, err)) return false;
  if (!read_layout(dir, old, old_segs, err)) return false;
  if (old.n < 1 || old.n > DP_MAX_N) return err.set(DP_ERR_IO, "checkpoint: saved layout has a bad n");
  std::vector<const ManifestEntry*> ents;
  for (const std::string& name : required_files(old.n)) {
    const ManifestEntry* e = nullptr;
    for (const ManifestEntry& x : man)
      if (x.name == name) e = &x;
    if (!e) return err.set(DP_ERR_IO, "checkpoint: manifest of " + dir + " lacks " + name);
    if (name == "user.bin" && user_bytes) *user_bytes = e->bytes;
    ents.push_back(e);
  }
  if (verify) {
    // one file per work item: the checksum chain is sequential within a file
    Err v = parallel_items((int64_t)ents.size(), io_workers(), [&](int64_t i, int, Err& e) {
      return verify_file(dir + "/" + ents[i]->name, *ents[i], e);
    });
    if (v.code != DP_OK) {
      err = v;
      return false;
    }
  }
  return true;
}

dp_status_t load(const char* root, const char* tag, const dp_layout_t* layout, float* const* master,
                 float* const* m, float* const* v, dp_step_state_t* d_state, void* user_meta,
                 uint64_t* user_meta_bytes, int32_t host_buffers, int32_t verify, cudaStream_t stream) {
  Err err;
  if (!root || !master || !m || !v || !d_state) return dp::report_error(DP_ERR_INVALID_ARG, "checkpoint: NULL argument");
  std::vector<Seg> nsegs, osegs;
  std::vector<int64_t> nlen, olen;
  if (!layout_segments(layout, nsegs, nlen, err)) return dp::report_error(err.code, err.msg.c_str());
  const bool full = layout->stage == DP_STAGE_DP;
  for (int r = 0; r < layout->n; ++r) {
    const int64_t need = full ? layout->psi : nlen[r];
    if (need && (!master[r] || !m[r] || !v[r]))
      return dp::report_error(DP_ERR_INVALID_ARG, "checkpoint: NULL state array of a non-empty shard");
  }
  std::string dir;
  dp_layout_t old;
  std::vector<dp_segment_t> old_segs;
  if (!open_checkpoint(root, tag, verify, dir, old, old_segs, nullptr, err)) return dp::report_error(err.code, err.msg.c_str());
  if (!layout_segments(&old, osegs, olen, err))
    return dp::report_error(DP_ERR_IO, "checkpoint: the saved layout is not valid");
  if (layout->psi != old.psi)
    return dp::report_error(DP_ERR_INVALID_ARG, "checkpoint: the parameter count differs from the saved one");

  if (!host_buffers) {
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return dp::report_error(DP_ERR_CUDA, cudaGetErrorString(e));
  }
  const int64_t cap = (int64_t)(CHUNK / sizeof(float));

  std::vector<int> fds(old.n, -1);
  for (int r = 0; r < old.n && err.code == DP_OK; ++r) {
    const std::string p = dir + "/shard_" + std::to_string(r) + ".bin";
    fds[r] = ::open(p.c_str(), O_RDONLY);
    if (fds[r] < 0) {
      err.set(DP_ERR_IO, "open " + p + ": " + strerror(errno));
      break;
    }
    uint32_t hdr[4];
    int64_t len = -1;
    struct stat fst;
    if (read_at(fds[r], hdr, sizeof(hdr), 0, err, p) && read_at(fds[r], &len, 8, 16, err, p) &&
        (hdr[0] != SHARD_MAGIC || hdr[1] != 1u || hdr[2] != (uint32_t)r || len != olen[r] ||
         ::fstat(fds[r], &fst) != 0 || fst.st_size != SHARD_HDR + 12 * olen[r]))
      err.set(DP_ERR_IO, "checkpoint: " + p + " does not match the saved layout");
  }
  // Reshard: each overlap of a new segment with an old one is a run of the same global elements; the runs,
  // cut into chunk-sized pieces for each of master/m/v, are the work items of the copy threads.
  struct Piece {
    int64_t lo, c;  // global start, elements
    int32_t k;      // 0 master, 1 m, 2 v
    int32_t ns, os;
  };
  // Both segment lists are sorted by global offset and tile [0, psi) without gaps, so one sweep over the two
  // finds every overlap (linear in the segment counts).
  std::vector<Piece> pieces;
  size_t b0 = 0;
  for (size_t a = 0; a < nsegs.size() && err.code == DP_OK; ++a) {
    const int64_t nend = nsegs[a].goff + nsegs[a].len;
    while (b0 < osegs.size() && osegs[b0].goff + osegs[b0].len <= nsegs[a].goff) ++b0;
    for (size_t b = b0; b < osegs.size() && osegs[b].goff < nend; ++b) {
      const int64_t lo = std::max(nsegs[a].goff, osegs[b].goff);
      const int64_t hi = std::min(nend, osegs[b].goff + osegs[b].len);
      for (int k = 0; k < 3; ++k)
        for (int64_t i = lo; i < hi; i += cap) pieces.push_back({i, std::min(hi - i, cap), k, (int32_t)a, (int32_t)b});
    }
  }
  float* const* arrays[3] = {master, m, v};
  if (err.code == DP_OK) {
    const int workers = io_workers();
    std::vector<Stager*> io;
    for (int k = 0; k < workers; ++k) io.push_back(new Stager(host_buffers));
    err = parallel_items((int64_t)pieces.size(), workers, [&](int64_t idx, int w, Err& e) {
      float* buf = io[w]->chunk(e);
      if (!buf) return false;
      const Piece& pc = pieces[idx];
      const Seg& ns = nsegs[pc.ns];
      const Seg& os = osegs[pc.os];
      const uint64_t off = (uint64_t)(SHARD_HDR + ((int64_t)pc.k * olen[os.owner] + os.loff + (pc.lo - os.goff)) * 4);
      if (!read_at(fds[os.owner], buf, (size_t)pc.c * 4, off, e, "shard")) return false;
      if (full) {
        // stage 0: every rank's full-length copy receives the element at its global index
        for (int r = 0; r < layout->n; ++r)
          if (!io[w]->in(arrays[pc.k][r] + pc.lo, buf, (size_t)pc.c * 4, e)) return false;
        return true;
      }
      return io[w]->in(arrays[pc.k][ns.owner] + ns.loff + (pc.lo - ns.goff), buf, (size_t)pc.c * 4, e);
    });
    for (Stager* x : io) delete x;
  }
  for (int fd : fds)
    if (fd >= 0) ::close(fd);
  Stager io(host_buffers, stream);  // the 64-byte state goes over the caller's stream
  if (err.code == DP_OK) {
    dp_step_state_t hs;
    int fd = ::open((dir + "/state.bin").c_str(), O_RDONLY);
    if (fd < 0) {
      err.set(DP_ERR_IO, "checkpoint: no state.bin in " + dir);
    } else {
      if (read_at(fd, &hs, sizeof(hs), 0, err, "state.bin")) io.in(d_state, &hs, sizeof(hs), err);
      ::close(fd);
    }
  }
  if (err.code == DP_OK && user_meta_bytes) {
    const std::string up = dir + "/user.bin";
    struct stat st;
    if (::stat(up.c_str(), &st) != 0) {
      err.set(DP_ERR_IO, "checkpoint: no user.bin in " + dir);
    } else {
      const uint64_t size = (uint64_t)st.st_size;
      if (user_meta && size > *user_meta_bytes) {
        err.set(DP_ERR_INVALID_ARG, "checkpoint: the user metadata is larger than the buffer");
      } else {
        if (user_meta && size) {
          int fd = ::open(up.c_str(), O_RDONLY);
          if (fd < 0) {
            err.set(DP_ERR_IO, "open " + up + ": " + strerror(errno));
          } else {
            read_at(fd, user_meta, (size_t)size, 0, err, "user.bin");
            ::close(fd);
          }
        }
        *user_meta_bytes = size;
      }
    }
  }
  if (err.code != DP_OK) return dp::report_error(err.code, err.msg.c_str());
  return DP_OK;
}

}  // namespace

extern "C" dp_status_t dp_checkpoint_save(const char* root, const char* tag, const dp_layout_t* layout,
                                          float* const* master, float* const* m, float* const* v,
                                          const dp_step_state_t* d_state, const void* user_meta,
                                          uint64_t user_meta_bytes, int32_t host_buffers, dp_stream_t stream) {
  return save(root, tag, layout, master, m, v, d_state, user_meta, user_meta_bytes, host_buffers,
              (cudaStream_t)stream);
}

extern "C" dp_status_t dp_checkpoint_load(const char* root, const char* tag, const dp_layout_t* layout,
                                          float* const* master, float* const* m, float* const* v,
                                          dp_step_state_t* d_state, void* user_meta, uint64_t* user_meta_bytes,
                                          int32_t host_buffers, int32_t verify, dp_stream_t stream) {
  return load(root, tag, layout, master, m, v, d_state, user_meta, user_meta_bytes, host_buffers, verify,
              (cudaStream_t)stream);
}

extern "C" dp_status_t dp_checkpoint_info(const char* root, const char* tag, int32_t verify, int32_t* stage,
                                          int32_t* n, int64_t* psi, int32_t* nseg, dp_segment_t* seg,
                                          int32_t seg_cap, uint64_t* user_meta_bytes) {
  Err err;
  if (!root) return dp::report_error(DP_ERR_INVALID_ARG, "checkpoint: NULL root");
  std::string dir;
  dp_layout_t old;
  std::vector<dp_segment_t> segs;
  if (!open_checkpoint(root, tag, verify, dir, old, segs, user_meta_bytes, err)) return dp::report_error(err.code, err.msg.c_str());
  if (stage) *stage = old.stage;
  if (n) *n = old.n;
  if (psi) *psi = old.psi;
  if (nseg) *nseg = old.nseg;
  if (seg) {
    if (seg_cap < old.nseg) return dp::report_error(DP_ERR_INVALID_ARG, "checkpoint: segment buffer too small");
    if (old.nseg) memcpy(seg, segs.data(), sizeof(dp_segment_t) * (size_t)old.nseg);
  }
  return DP_OK;
}
