// Seeded synthetic workload generators: graphs (CSR, destination-major) and
// feature arrays.  This file holds none of the aggregation arithmetic; it only
// draws inputs.  Every random number comes from a counter-based generator
// (splitmix64 of a seeded key and an index), so a result never depends on the
// number of threads that produced it.
//
// CSR convention: row i lists the sources j of the edges j -> i, sorted
// ascending, duplicates removed, with exactly one self-loop per node.

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <numeric>
#include <thread>
#include <vector>

namespace {

inline uint64_t mix64(uint64_t x) {
  // splitmix64 finaliser (Steele, Lea, Flood: "Fast splittable pseudorandom
  // number generators", OOPSLA 2014).
  x += 0x9e3779b97f4a7c15ULL;
  x = (x ^ (x >> 30)) * 0xbf58476d1ce4e5b9ULL;
  x = (x ^ (x >> 27)) * 0x94d049bb133111ebULL;
  return x ^ (x >> 31);
}

struct Stream {
  uint64_t key;
  Stream(uint64_t seed, uint64_t stream) : key(mix64(mix64(seed) ^ (stream * 0xd1342543de82ef95ULL))) {}
  uint64_t at(uint64_t idx) const { return mix64(key + idx * 0x9e3779b97f4a7c15ULL); }
  // uniform double in [0, 1)
  double u01(uint64_t idx) const { return double(at(idx) >> 11) * 0x1.0p-53; }
  // uniform double in (0, 1]
  double u01_open0(uint64_t idx) const { return double((at(idx) >> 11) + 1) * 0x1.0p-53; }
};

int n_threads() {
  const char* env = std::getenv("GNN_GEN_THREADS");
  if (env && std::atoi(env) > 0) return std::atoi(env);
  unsigned hc = std::thread::hardware_concurrency();
  return hc ? int(std::min(hc, 64u)) : 4;
}

template <typename F>
void parallel_for(int64_t n, F&& f) {
  int T = n_threads();
  if (n < 4096 || T <= 1) {
    f(int64_t(0), n, 0);
    return;
  }
  std::vector<std::thread> ts;
  int64_t per = (n + T - 1) / T;
  for (int t = 0; t < T; ++t) {
    int64_t b = t * per, e = std::min(n, b + per);
    if (b >= e) break;
    ts.emplace_back([&f, b, e, t] { f(b, e, t); });
  }
  for (auto& t : ts) t.join();
}

struct Graph {
  int64_t n = 0;
  std::vector<int32_t> row_ptr;  // n + 1
  std::vector<int32_t> col;      // E
};

// Build a CSR from (dst, src) pairs: add one self-loop per node, sort each row,
// drop duplicates.  Pairs with dst == src are dropped first (the self-loop that
// is added replaces them).
Graph build_csr(int64_t n, const std::vector<int32_t>& dst, const std::vector<int32_t>& src) {
  const int64_t m = int64_t(dst.size());
  std::vector<std::atomic<int32_t>> cnt(n);
  for (int64_t i = 0; i < n; ++i) cnt[i].store(1, std::memory_order_relaxed);  // the self-loop
  parallel_for(m, [&](int64_t b, int64_t e, int) {
    for (int64_t k = b; k < e; ++k)
      if (dst[k] != src[k]) cnt[dst[k]].fetch_add(1, std::memory_order_relaxed);
  });
  std::vector<int64_t> off(n + 1, 0);
  for (int64_t i = 0; i < n; ++i) off[i + 1] = off[i] + cnt[i].load(std::memory_order_relaxed);
  std::vector<int32_t> tmp(off[n]);
  std::vector<std::atomic<int64_t>> cur(n);
  for (int64_t i = 0; i < n; ++i) {
    tmp[off[i]] = int32_t(i);
    cur[i].store(off[i] + 1, std::memory_order_relaxed);
  }
  parallel_for(m, [&](int64_t b, int64_t e, int) {
    for (int64_t k = b; k < e; ++k)
      if (dst[k] != src[k]) tmp[cur[dst[k]].fetch_add(1, std::memory_order_relaxed)] = src[k];
  });
  // sort + unique per row (the scatter order above is irrelevant after this)
  std::vector<int32_t> len(n);
  parallel_for(n, [&](int64_t b, int64_t e, int) {
    for (int64_t i = b; i < e; ++i) {
      int32_t* p = tmp.data() + off[i];
      int32_t* q = tmp.data() + off[i + 1];
      std::sort(p, q);
      len[i] = int32_t(std::unique(p, q) - p);
    }
  });
  Graph g;
  g.n = n;
  g.row_ptr.assign(n + 1, 0);
  for (int64_t i = 0; i < n; ++i) g.row_ptr[i + 1] = g.row_ptr[i] + len[i];
  g.col.resize(g.row_ptr[n]);
  parallel_for(n, [&](int64_t b, int64_t e, int) {
    for (int64_t i = b; i < e; ++i)
      std::memcpy(g.col.data() + g.row_ptr[i], tmp.data() + off[i], sizeof(int32_t) * len[i]);
  });
  return g;
}

// Fisher-Yates permutation of [0, n) driven by the counter-based stream.
std::vector<int32_t> permutation(int64_t n, const Stream& s) {
  std::vector<int32_t> p(n);
  std::iota(p.begin(), p.end(), 0);
  for (int64_t i = n - 1; i > 0; --i) {
    uint64_t r = s.at(uint64_t(i));
    int64_t j = int64_t((unsigned __int128)r * uint64_t(i + 1) >> 64);
    std::swap(p[i], p[j]);
  }
  return p;
}

Graph relabel(const Graph& g, const std::vector<int32_t>& new_id) {
  const int64_t n = g.n, E = int64_t(g.col.size());
  std::vector<int32_t> dst(E), src(E);
  parallel_for(n, [&](int64_t b, int64_t e, int) {
    for (int64_t i = b; i < e; ++i)
      for (int64_t k = g.row_ptr[i]; k < g.row_ptr[i + 1]; ++k) {
        dst[k] = new_id[i];
        src[k] = new_id[g.col[k]];
      }
  });
  return build_csr(n, dst, src);
}

}  // namespace

struct gen_graph {
  Graph g;
};

extern "C" {

// ---- features -------------------------------------------------------------

// Normal(0, std) samples by Box-Muller; element k uses the pair k/2 of the
// stream (cos for even k, sin for odd k).
void gen_normal_f32(uint64_t seed, uint64_t stream, int64_t n, double std_dev, float* out) {
  Stream s(seed, stream);
  parallel_for((n + 1) / 2, [&](int64_t b, int64_t e, int) {
    for (int64_t k = b; k < e; ++k) {
      double u1 = s.u01_open0(2 * uint64_t(k));
      double u2 = s.u01(2 * uint64_t(k) + 1);
      double r = std::sqrt(-2.0 * std::log(u1));
      double t = 6.283185307179586476925286766559 * u2;
      out[2 * k] = float(std_dev * r * std::cos(t));
      if (2 * k + 1 < n) out[2 * k + 1] = float(std_dev * r * std::sin(t));
    }
  });
}

// Round float32 to bfloat16 (round to nearest, ties to even; NaN kept quiet).
void gen_f32_to_bf16(int64_t n, const float* in, uint16_t* out) {
  parallel_for(n, [&](int64_t b, int64_t e, int) {
    for (int64_t k = b; k < e; ++k) {
      uint32_t u;
      std::memcpy(&u, in + k, 4);
      if ((u & 0x7fffffffu) > 0x7f800000u) {
        out[k] = uint16_t((u >> 16) | 0x40u);
      } else {
        uint32_t lsb = (u >> 16) & 1u;
        out[k] = uint16_t((u + 0x7fffu + lsb) >> 16);
      }
    }
  });
}

// ---- graphs ---------------------------------------------------------------

int64_t gen_graph_nodes(const gen_graph* h) { return h ? h->g.n : -1; }
int64_t gen_graph_edges(const gen_graph* h) { return h ? int64_t(h->g.col.size()) : -1; }
void gen_graph_copy(const gen_graph* h, int32_t* row_ptr, int32_t* col) {
  std::memcpy(row_ptr, h->g.row_ptr.data(), sizeof(int32_t) * (h->g.n + 1));
  std::memcpy(col, h->g.col.data(), sizeof(int32_t) * h->g.col.size());
}
void gen_graph_free(gen_graph* h) { delete h; }

// Wrap an existing CSR (copied) so it can be relabelled.
gen_graph* gen_graph_from_csr(int64_t n, const int32_t* row_ptr, const int32_t* col) {
  auto* h = new gen_graph;
  h->g.n = n;
  h->g.row_ptr.assign(row_ptr, row_ptr + n + 1);
  h->g.col.assign(col, col + row_ptr[n]);
  return h;
}

// Erdos-Renyi: every ordered pair j -> i, j != i, kept with p = avg / (n - 1);
// candidates are visited with geometric skips.  One self-loop per node.
gen_graph* gen_graph_er(int64_t n, double avg_deg, uint64_t seed) {
  if (n <= 0) return nullptr;
  double p = n > 1 ? std::min(1.0, avg_deg / double(n - 1)) : 0.0;
  std::vector<std::vector<int32_t>> rows(n);
  parallel_for(n, [&](int64_t b, int64_t e, int) {
    for (int64_t i = b; i < e; ++i) {
      Stream s(seed, 0x1000000ULL + uint64_t(i));
      if (p <= 0.0) continue;
      const double lq = std::log1p(-p);
      int64_t j = -1;
      uint64_t draw = 0;
      for (;;) {
        double u = s.u01_open0(draw++);
        int64_t skip = (p >= 1.0) ? 0 : int64_t(std::floor(std::log(u) / lq));
        j += 1 + skip;
        if (j >= n - 1) break;
        int64_t src = j < i ? j : j + 1;  // candidates exclude i itself
        rows[i].push_back(int32_t(src));
      }
    }
  });
  std::vector<int32_t> dst, src;
  for (int64_t i = 0; i < n; ++i)
    for (int32_t j : rows[i]) {
      dst.push_back(int32_t(i));
      src.push_back(j);
    }
  auto* h = new gen_graph;
  h->g = build_csr(n, dst, src);
  return h;
}

// Every node gets `k` distinct sources != i, uniform without replacement,
// plus its self-loop (in-degree exactly k + 1 when n > k).
gen_graph* gen_graph_uniform(int64_t n, int64_t k, uint64_t seed) {
  if (n <= 0 || k < 0) return nullptr;
  k = std::min<int64_t>(k, n - 1);
  std::vector<int32_t> dst(n * k), src(n * k);
  parallel_for(n, [&](int64_t b, int64_t e, int) {
    std::vector<int32_t> pick;
    for (int64_t i = b; i < e; ++i) {
      Stream s(seed, 0x2000000ULL + uint64_t(i));
      pick.clear();
      uint64_t draw = 0;
      while (int64_t(pick.size()) < k) {
        int64_t j = int64_t((unsigned __int128)s.at(draw++) * uint64_t(n - 1) >> 64);
        if (j >= i) ++j;
        if (std::find(pick.begin(), pick.end(), int32_t(j)) == pick.end()) pick.push_back(int32_t(j));
      }
      for (int64_t t = 0; t < k; ++t) {
        dst[i * k + t] = int32_t(i);
        src[i * k + t] = pick[t];
      }
    }
  });
  auto* h = new gen_graph;
  h->g = build_csr(n, dst, src);
  return h;
}

// Chung-Lu with power-law weights w_r = c (r + 1)^(-1/(gamma-1)), capped at
// `cap`, c chosen so that the mean weight is `avg`.  n*avg endpoint pairs are
// drawn with dst ~ w and src ~ w independently; node ids are a seeded
// permutation of the weight ranks.
gen_graph* gen_graph_chung_lu(int64_t n, double gamma, double avg, double cap, uint64_t seed) {
  if (n <= 1 || gamma <= 1.0 || avg <= 0.0) return nullptr;
  const double beta = 1.0 / (gamma - 1.0);
  std::vector<double> base(n);
  for (int64_t r = 0; r < n; ++r) base[r] = std::pow(double(r + 1), -beta);
  auto mean_for = [&](double c) {
    double s = 0.0;
    for (int64_t r = 0; r < n; ++r) s += std::min(cap, c * base[r]);
    return s / double(n);
  };
  double lo = 0.0, hi = 1.0;
  while (mean_for(hi) < avg && hi < 1e300) hi *= 2.0;
  for (int it = 0; it < 100; ++it) {
    double mid = 0.5 * (lo + hi);
    (mean_for(mid) < avg ? lo : hi) = mid;
  }
  const double c = 0.5 * (lo + hi);
  std::vector<double> cdf(n + 1, 0.0);
  for (int64_t r = 0; r < n; ++r) cdf[r + 1] = cdf[r] + std::min(cap, c * base[r]);
  const double total = cdf[n];
  auto sample = [&](double u) {
    double x = u * total;
    int64_t r = int64_t(std::upper_bound(cdf.begin(), cdf.end(), x) - cdf.begin()) - 1;
    return std::min<int64_t>(std::max<int64_t>(r, 0), n - 1);
  };
  std::vector<int32_t> perm = permutation(n, Stream(seed, 0x3000001ULL));
  const int64_t m = int64_t(std::llround(double(n) * avg));
  std::vector<int32_t> dst(m), src(m);
  Stream sd(seed, 0x3000002ULL), ss(seed, 0x3000003ULL);
  parallel_for(m, [&](int64_t b, int64_t e, int) {
    for (int64_t k = b; k < e; ++k) {
      dst[k] = perm[sample(sd.u01(uint64_t(k)))];
      src[k] = perm[sample(ss.u01(uint64_t(k)))];
    }
  });
  auto* h = new gen_graph;
  h->g = build_csr(n, dst, src);
  return h;
}

// R-MAT (Chakrabarti, Zhan, Faloutsos 2004): 2^scale nodes, edge_factor * 2^scale
// samples, each by `scale` quadrant choices with probabilities (a, b, c, d);
// the quadrant's row bit goes to the destination, its column bit to the source.
gen_graph* gen_graph_rmat(int scale, int64_t edge_factor, double a, double b, double c, uint64_t seed) {
  if (scale < 1 || scale > 30 || edge_factor < 1) return nullptr;
  const int64_t n = int64_t(1) << scale;
  const int64_t m = n * edge_factor;
  std::vector<int32_t> dst(m), src(m);
  Stream s(seed, 0x4000001ULL);
  const double ab = a + b, abc = a + b + c;
  parallel_for(m, [&](int64_t lo, int64_t hi, int) {
    for (int64_t k = lo; k < hi; ++k) {
      int64_t row = 0, colv = 0;
      for (int l = 0; l < scale; ++l) {
        double u = s.u01(uint64_t(k) * uint64_t(scale) + uint64_t(l));
        int rb, cb;
        if (u < a) { rb = 0; cb = 0; }
        else if (u < ab) { rb = 0; cb = 1; }
        else if (u < abc) { rb = 1; cb = 0; }
        else { rb = 1; cb = 1; }
        row = (row << 1) | rb;
        colv = (colv << 1) | cb;
      }
      dst[k] = int32_t(row);
      src[k] = int32_t(colv);
    }
  });
  auto* h = new gen_graph;
  h->g = build_csr(n, dst, src);
  return h;
}

// Relabel with a seeded random permutation (the "random node ids" variant).
gen_graph* gen_graph_permute_random(const gen_graph* in, uint64_t seed) {
  if (!in) return nullptr;
  std::vector<int32_t> p = permutation(in->g.n, Stream(seed, 0x5000001ULL));
  auto* h = new gen_graph;
  h->g = relabel(in->g, p);
  return h;
}

// Reverse Cuthill-McKee order on the symmetrised graph (self-loops ignored).
// Each component starts at the unvisited node of smallest degree (ties: lower
// id); a node's unvisited neighbours are enqueued by ascending degree (ties:
// lower id).  new_id[v] = position of v in the reversed visit order.
void gen_rcm_order(const gen_graph* in, int32_t* new_id) {
  const Graph& g = in->g;
  const int64_t n = g.n;
  // symmetrised adjacency without self-loops, deduplicated
  std::vector<int32_t> dst, src;
  dst.reserve(g.col.size() * 2);
  src.reserve(g.col.size() * 2);
  for (int64_t i = 0; i < n; ++i)
    for (int64_t k = g.row_ptr[i]; k < g.row_ptr[i + 1]; ++k) {
      int32_t j = g.col[k];
      if (j == i) continue;
      dst.push_back(int32_t(i)); src.push_back(j);
      dst.push_back(j); src.push_back(int32_t(i));
    }
  Graph s = build_csr(n, dst, src);  // adds self-loops: skipped below
  std::vector<int32_t> deg(n);
  for (int64_t i = 0; i < n; ++i) deg[i] = s.row_ptr[i + 1] - s.row_ptr[i] - 1;
  std::vector<int32_t> by_deg(n);
  std::iota(by_deg.begin(), by_deg.end(), 0);
  std::stable_sort(by_deg.begin(), by_deg.end(), [&](int32_t x, int32_t y) { return deg[x] < deg[y]; });
  std::vector<char> seen(n, 0);
  std::vector<int32_t> order;
  order.reserve(n);
  std::vector<int32_t> nb;
  int64_t next = 0;
  while (int64_t(order.size()) < n) {
    while (seen[by_deg[next]]) ++next;
    int32_t start = by_deg[next];
    seen[start] = 1;
    size_t head = order.size();
    order.push_back(start);
    while (head < order.size()) {
      int32_t v = order[head++];
      nb.clear();
      for (int64_t k = s.row_ptr[v]; k < s.row_ptr[v + 1]; ++k) {
        int32_t w = s.col[k];
        if (w != v && !seen[w]) { seen[w] = 1; nb.push_back(w); }
      }
      std::sort(nb.begin(), nb.end(), [&](int32_t x, int32_t y) {
        return deg[x] != deg[y] ? deg[x] < deg[y] : x < y;
      });
      order.insert(order.end(), nb.begin(), nb.end());
    }
  }
  for (int64_t k = 0; k < n; ++k) new_id[order[n - 1 - k]] = int32_t(k);
}

gen_graph* gen_graph_relabel(const gen_graph* in, const int32_t* new_id) {
  if (!in) return nullptr;
  std::vector<int32_t> p(new_id, new_id + in->g.n);
  auto* h = new gen_graph;
  h->g = relabel(in->g, p);
  return h;
}

}  // extern "C"
