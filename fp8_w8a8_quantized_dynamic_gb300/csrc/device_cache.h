// Per-device memo for launch-configuration facts (kernel attributes set, co-resident cluster
// counts, shared-memory limits). One process may drive several GPUs from several host threads,
// so every entry is keyed by the device ordinal as well as its own key, and the table is
// guarded by a mutex. A value is stored only when it was computed successfully, so a failed
// query is retried on the next call instead of being remembered.
#pragma once

#include <cstddef>
#include <map>
#include <mutex>
#include <utility>

namespace fp8k {

template <typename Key, typename Value>
class PerDeviceCache {
 public:
  // The value for (device, key): the stored one, or compute(&value) -> bool on first use.
  template <typename Fn>
  bool get(int device, const Key& key, Value* out, Fn&& compute) {
    std::lock_guard<std::mutex> g(mu_);
    const auto k = std::make_pair(device, key);
    auto it = map_.find(k);
    if (it != map_.end()) {
      *out = it->second;
      return true;
    }
    Value v{};
    if (!compute(&v)) return false;
    map_.emplace(k, v);
    *out = v;
    return true;
  }

  size_t size() {
    std::lock_guard<std::mutex> g(mu_);
    return map_.size();
  }

 private:
  std::mutex mu_;
  std::map<std::pair<int, Key>, Value> map_;
};

}  // namespace fp8k
