"""GB300-native sparse offloaded-KV decode step (landmark top-k selection,
predicted-vs-needed diff, coalesced host->HBM gather into a two-layer ping-pong
buffer, GQA decode attention with a log-sum-exp window merge)."""
