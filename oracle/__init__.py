"""fp64 CPU oracle for split-KV paged attention (test infrastructure only)."""
