"""GB300-native DSA sparse-attention decode (k-pooled indexer + sparse latent MLA)."""
