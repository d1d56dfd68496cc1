"""CPU oracle (test infrastructure only): see ``oracle.llama_oracle``."""
